"""C-ABI checks that need no GPU: the library loads, exports every declared entry point,
its struct layouts match the Python binding, and host-side validation rejects bad calls
(before any launch) with the documented status codes."""
import ctypes
import os
import re
import subprocess

import pytest

import long_context_sparse_tcgen05_gb300 as dsa
from long_context_sparse_tcgen05_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, SCHEDULE = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"dsa_indexer_scores", "dsa_topk", "dsa_sparse_attn", "indexshare_group_forward",
            "topk_overlap"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dsa.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(dsa_indexer_args),'
                   ' sizeof(dsa_attn_args), sizeof(dsa_topk_src), sizeof(dsa_layer),'
                   ' offsetof(dsa_indexer_args, q_pos0), offsetof(dsa_attn_args, q),'
                   ' offsetof(dsa_layer, out)); return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(dsa.IndexerArgs), ctypes.sizeof(dsa.AttnArgs), ctypes.sizeof(dsa.TopkSrc),
            ctypes.sizeof(dsa.Layer), dsa.IndexerArgs.q_pos0.offset, dsa.AttnArgs.q.offset,
            dsa.Layer.out.offset]
    assert got == want


def test_status_strings(lib):
    assert dsa.status_string(0) == "DSA_OK"
    assert dsa.status_string(5) == "DSA_ERR_SCHEDULE"


# Fake, 16-byte aligned "device" addresses: validation must fail before any launch, so
# nothing ever dereferences them.
FAKE = 0x10000000


def _ix(**kw):
    a = dsa.IndexerArgs(1, 64, 64, 64, 128, dsa.DSA_BF16, FAKE, None, FAKE, FAKE, None, 0, 0)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _at(**kw):
    a = dsa.AttnArgs(1, 64, 64, 64, 576, 512, 0.04, FAKE, FAKE, 576, FAKE, 576)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _topk_ix(lib, ix, k=16, ws=FAKE, ws_bytes=1 << 30, **over):
    src = dsa.TopkSrc(dsa.TOPK_FROM_INDEXER, None, 0, ctypes.pointer(ix))
    args = dict(B=ix.B, T=ix.T, S=ix.S, q_pos0=ix.q_pos0, diag=ix.diag)
    args.update(over)
    return lib.dsa_topk(ctypes.byref(src), args["B"], args["T"], args["S"], args["q_pos0"], args["diag"],
                        k, ctypes.c_void_p(FAKE), ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("field,value,status", [
    ("B", 0, INVALID), ("T", -1, INVALID), ("H_I", 32, UNSUPPORTED), ("d_I", 96, UNSUPPORTED),
    ("q", None, INVALID), ("q", FAKE + 4, MISALIGNED), ("k", FAKE + 8, MISALIGNED),
    ("diag", 2, INVALID), ("q_pos0", -5, INVALID), ("dtype", 7, INVALID),
])
def test_topk_indexer_arg_validation(lib, field, value, status):
    ix = _ix(**{field: value})
    assert _topk_ix(lib, ix) == status
    assert dsa.load_library().dsa_last_error().decode()


def test_topk_e4m3_needs_scales(lib):
    assert _topk_ix(lib, _ix(dtype=dsa.DSA_E4M3)) == INVALID
    assert _topk_ix(lib, _ix(dtype=dsa.DSA_E4M3, H_I=4, d_I=64, q_scale=FAKE, k_scale=FAKE)) == UNSUPPORTED


@pytest.mark.parametrize("k", [0, -1, 4097])
def test_topk_k_range(lib, k):
    assert _topk_ix(lib, _ix(), k=k) == UNSUPPORTED


def test_topk_shape_mismatch_and_workspace(lib):
    assert _topk_ix(lib, _ix(), T=32) == INVALID
    assert _topk_ix(lib, _ix(), ws=0) == WORKSPACE
    assert _topk_ix(lib, _ix(), ws=FAKE + 8) == MISALIGNED
    assert _topk_ix(lib, _ix(), ws_bytes=100) == WORKSPACE
    assert _topk_ix(lib, _ix(), ws_bytes=300) == WORKSPACE  # not even one score row


def test_topk_scores_validation(lib):
    src = dsa.TopkSrc(dsa.TOPK_FROM_SCORES, None, 64, None)
    assert lib.dsa_topk(ctypes.byref(src), 1, 4, 64, 0, 0, 8, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 20, None) == INVALID
    src = dsa.TopkSrc(dsa.TOPK_FROM_SCORES, FAKE, 32, None)
    assert lib.dsa_topk(ctypes.byref(src), 1, 4, 64, 0, 0, 8, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 20, None) == INVALID
    src = dsa.TopkSrc(9, FAKE, 64, None)
    assert lib.dsa_topk(ctypes.byref(src), 1, 4, 64, 0, 0, 8, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 20, None) == INVALID


@pytest.mark.parametrize("field,value,status", [
    ("H", 32, UNSUPPORTED), ("d_qk", 128, UNSUPPORTED), ("q", None, INVALID), ("k", FAKE + 2, MISALIGNED),
    ("k_ld", 570, MISALIGNED), ("v_ld", 100, MISALIGNED), ("scale", 0.0, INVALID), ("S", 0, INVALID),
])
def test_attention_arg_validation(lib, field, value, status):
    at = _at(**{field: value})
    r = lib.dsa_sparse_attn(ctypes.byref(at), ctypes.c_void_p(FAKE), 16, ctypes.c_void_p(FAKE), None,
                            ctypes.c_void_p(FAKE), 256, None)
    assert r == status


def test_attention_null_idx_and_bad_k(lib):
    at = _at()
    assert lib.dsa_sparse_attn(ctypes.byref(at), None, 16, ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE), 256, None) == INVALID
    assert lib.dsa_sparse_attn(ctypes.byref(at), ctypes.c_void_p(FAKE), 0, ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE), 256, None) == UNSUPPORTED
    assert lib.dsa_sparse_attn(ctypes.byref(at), ctypes.c_void_p(FAKE), 16, ctypes.c_void_p(FAKE + 2), None, ctypes.c_void_p(FAKE), 256, None) == MISALIGNED


def _group(lib, schedule, n_layers=4, ws_bytes=1 << 30, bufs=True, layer_edit=None):
    arr = (dsa.Layer * n_layers)()
    for i in range(n_layers):
        arr[i].ix = _ix()
        arr[i].at = _at()
        arr[i].out = FAKE
        arr[i].lse = None
    if layer_edit:
        layer_edit(arr)
    b = (ctypes.c_void_p * 4)(FAKE, FAKE, FAKE, FAKE)
    sched = None if schedule is None else schedule.encode()
    return lib.indexshare_group_forward(arr, n_layers, sched, 16, b if bufs else None,
                                        ctypes.c_void_p(FAKE), ws_bytes, None)


@pytest.mark.parametrize("schedule", ["SFSS", "FSS", "FSSSS", "FSXS", "", "fsss", None])
def test_group_schedule_validation(lib, schedule):
    assert _group(lib, schedule) == SCHEDULE


def test_group_layer_validation(lib):
    def bad_at(arr):
        arr[2].at.H = 3
    assert _group(lib, "FSSS", layer_edit=bad_at) == UNSUPPORTED

    def bad_ix_in_f(arr):
        arr[0].ix.d_I = 3
    assert _group(lib, "FSSS", layer_edit=bad_ix_in_f) == UNSUPPORTED

    def bad_ix_in_s(arr):  # shared layers' indexer args are ignored
        arr[1].ix.d_I = 3
        arr[1].at.T = 64
    assert _group(lib, "FSSS", layer_edit=bad_ix_in_s, ws_bytes=100) == WORKSPACE

    def mismatched(arr):
        arr[3].at.T = 8
    assert _group(lib, "FSSS", layer_edit=mismatched) == INVALID
    assert _group(lib, "FSSS", bufs=False) == INVALID
    assert _group(lib, "FSSS", ws_bytes=300) == WORKSPACE


def test_overlap_validation(lib):
    m = ctypes.c_double()
    assert lib.topk_overlap(None, ctypes.c_void_p(FAKE), 4, 8, None, ctypes.byref(m), ctypes.c_void_p(FAKE), 1 << 20, None) == INVALID
    assert lib.topk_overlap(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 4, 0, None, ctypes.byref(m), ctypes.c_void_p(FAKE), 1 << 20, None) == INVALID
    assert lib.topk_overlap(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1000, 8, None, ctypes.byref(m), ctypes.c_void_p(FAKE), 300, None) == WORKSPACE


def test_workspace_size_plan(lib):
    ix = _ix(T=131072, S=131072)
    n = lib.dsa_workspace_size(ctypes.byref(ix), 2048)
    # a score chunk of at most 4 GiB, plus the candidate lists of the selecting path (at most
    # 1 GiB: 8,192 keys and positions per row of a chunk)
    assert n >= 256 + 131072 * 4 and n <= 256 + (4 << 30) + (1 << 30)
    assert n > 256 + (4 << 30)  # 64 heads, k = 2,048, many rows: the selecting path applies
    # k beyond the selecting path, or 4 indexer heads: the score chunk alone
    assert lib.dsa_workspace_size(ctypes.byref(ix), 4096) <= 256 + (4 << 30)
    small = _ix(T=131072, S=131072, H_I=4, d_I=64)
    assert lib.dsa_workspace_size(ctypes.byref(small), 64) <= 256 + (4 << 30)
    assert lib.dsa_workspace_size(None, 16) == 256


def test_trace_enable_validation_and_empty_read(lib):
    assert lib.dsa_trace_enable(0) == INVALID
    assert lib.dsa_trace_enable(-5) == INVALID
    assert lib.dsa_trace_enable((1 << 20) + 1) == INVALID
    dropped = ctypes.c_int32(7)
    # nothing recorded: no records, no drops, nothing dereferenced in the null arrays
    assert lib.dsa_trace_read(None, None, 0, ctypes.byref(dropped)) == 0
    assert dropped.value == 0
    lib.dsa_trace_disable()


def test_overlap_matrix_validation(lib):
    P = ctypes.c_void_p
    m = (ctypes.c_double * 256)()
    bufs = (P * 16)(*([FAKE] * 16))
    need4 = lib.topk_overlap_matrix_workspace_size(4)
    assert need4 == 256 + 8 * (16 * 16 + 1024 * 16)

    def call(b, n, rows, k, ws_bytes, out=m):
        return lib.topk_overlap_matrix(b, n, rows, k, None, out, P(FAKE), ws_bytes, None)

    assert call(None, 4, 10, 8, need4) == INVALID
    assert call(bufs, 4, 10, 8, need4, out=None) == INVALID
    assert call(bufs, 0, 10, 8, need4) == INVALID
    assert call(bufs, 17, 10, 8, 1 << 30) == INVALID
    assert call(bufs, 4, -1, 8, need4) == INVALID
    assert call(bufs, 4, 10, 0, need4) == INVALID
    assert call((P * 4)(FAKE, None, FAKE, FAKE), 4, 10, 8, need4) == INVALID
    # one CTA holds a row of every buffer: 16 x 3,072 fits, 16 x 4,096 does not, 12 x 4,096 does
    assert call(bufs, 16, 10, 4096, 1 << 30) == UNSUPPORTED
    assert call(bufs, 4, 10, 8, need4 - 8) == WORKSPACE
    assert call(bufs, 16, 10, 3072, lib.topk_overlap_matrix_workspace_size(16) - 1) == WORKSPACE
    assert call(bufs, 12, 10, 4096, lib.topk_overlap_matrix_workspace_size(12) - 1) == WORKSPACE


def test_schedule_validation(lib):
    M = [[1.0, 0.5], [0.5, 1.0]]
    with pytest.raises(dsa.DsaError) as e:
        dsa.indexshare_schedule_score(M, "SF")
    assert e.value.status == SCHEDULE
    for bad in ("F", "FSS", "FX"):
        with pytest.raises(dsa.DsaError):
            dsa.indexshare_schedule_score(M, bad)
    for n_full in (0, 3):
        with pytest.raises(dsa.DsaError) as e:
            dsa.indexshare_schedule_search(M, n_full)
        assert e.value.status == INVALID


def test_quantize_append_validation(lib):
    P = ctypes.c_void_p

    def call(x=FAKE, B=2, n=3, width=128, stride=384, codes=FAKE, scales=FAKE, S_cap=10, pos0=0,
             positions=None, ws_bytes=1 << 20):
        return lib.dsa_quantize_e4m3_append(P(x) if x else None, B, n, width, stride, P(codes) if codes else None,
                                            P(scales) if scales else None, S_cap, pos0,
                                            P(positions) if positions else None, P(FAKE), ws_bytes, None)

    assert call(x=0) == INVALID
    assert call(codes=0) == INVALID
    assert call(scales=0) == INVALID
    assert call(B=0) == INVALID
    assert call(S_cap=0) == INVALID
    assert call(width=130, stride=390) == UNSUPPORTED
    assert call(width=65540, stride=3 * 65540) == UNSUPPORTED
    assert call(stride=383) == INVALID
    assert call(x=FAKE + 4) == MISALIGNED
    assert call(stride=386) == MISALIGNED
    assert call(codes=FAKE + 2) == MISALIGNED
    assert call(pos0=8) == INVALID          # rows 8..10 do not fit 10
    assert call(pos0=-1) == INVALID
    assert call(ws_bytes=100) == WORKSPACE


def test_varlen_struct_layout(tmp_path):
    src = tmp_path / "vl.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dsa.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu\\n", sizeof(dsa_varlen), offsetof(dsa_varlen, cu_q),'
                   ' offsetof(dsa_varlen, cu_k), offsetof(dsa_varlen, q_pos0)); return 0;}\n')
    exe = tmp_path / "vl"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    assert got == [ctypes.sizeof(dsa.Varlen), dsa.Varlen.cu_q.offset, dsa.Varlen.cu_k.offset,
                   dsa.Varlen.q_pos0.offset]


def _varlen(lib, cu_q, cu_k, q_pos0, schedule="FSSS", T=None, S=None, layer_edit=None, seqs=True, ws_bytes=1 << 30):
    n_layers = len(schedule) if schedule else 4
    arr = (dsa.Layer * n_layers)()
    for i in range(n_layers):
        arr[i].ix = _ix(T=T if T is not None else cu_q[-1], S=S if S is not None else cu_k[-1])
        arr[i].at = _at(T=T if T is not None else cu_q[-1], S=S if S is not None else cu_k[-1])
        arr[i].out = FAKE
        arr[i].lse = None
    if layer_edit:
        layer_edit(arr)
    n = len(q_pos0)
    v = dsa.Varlen(n, (ctypes.c_int64 * len(cu_q))(*cu_q), (ctypes.c_int64 * len(cu_k))(*cu_k),
                   (ctypes.c_int64 * max(1, n))(*q_pos0))
    b = (ctypes.c_void_p * 4)(FAKE, FAKE, FAKE, FAKE)
    return lib.indexshare_group_forward_varlen(arr, n_layers, schedule.encode() if schedule else None, 16,
                                               ctypes.byref(v) if seqs else None, b, ctypes.c_void_p(FAKE),
                                               ws_bytes, None)


def test_varlen_validation(lib):
    ok = ([0, 64, 96], [0, 64, 160], [0, 32])
    assert _varlen(lib, *ok, seqs=False) == INVALID
    assert _varlen(lib, [4, 64, 96], [0, 64, 160], [0, 32]) == INVALID      # cu_q[0] != 0
    assert _varlen(lib, [0, 64, 60], [0, 64, 160], [0, 32]) == INVALID      # decreasing
    assert _varlen(lib, [0, 64, 96], [0, 64, 64], [0, 32]) == INVALID       # a sequence with no key
    assert _varlen(lib, *ok, T=100) == INVALID                              # packed rows != cu_q[n]
    assert _varlen(lib, *ok, S=100) == INVALID
    assert _varlen(lib, *ok, schedule="FSS") != OK and _varlen(lib, *ok, schedule="SFSS") == SCHEDULE

    def odd_k(arr):  # key rows of 64 bf16 values: sequence 1 starts 64 rows in, 16-byte aligned
        for i in range(4):
            arr[i].at.H = 3
    assert _varlen(lib, *ok, layer_edit=odd_k) == UNSUPPORTED
    # a sequence whose q_pos0 leaves its last rows without a key in the cache
    assert _varlen(lib, *ok[:2], [0, -1]) == INVALID
    assert _varlen(lib, *ok, ws_bytes=300) == WORKSPACE


def test_varlen_workspace_is_the_largest_sequence_need(lib):
    cu = [0, 1000, 1000 + 131072, 1000 + 131072 + 5]
    v = dsa.Varlen(3, (ctypes.c_int64 * 4)(*cu), (ctypes.c_int64 * 4)(*cu), (ctypes.c_int64 * 3)(0, 0, 0))
    ix = _ix(T=cu[-1], S=cu[-1])
    got = lib.dsa_workspace_size_varlen(ctypes.byref(ix), ctypes.byref(v), 2048)
    want = 0
    for b in range(3):
        one = _ix(T=cu[b + 1] - cu[b], S=cu[b + 1] - cu[b])
        want = max(want, lib.dsa_workspace_size(ctypes.byref(one), 2048))
    assert got == want
    # malformed sequences fall back to the minimum
    bad = dsa.Varlen(1, (ctypes.c_int64 * 2)(3, 9), (ctypes.c_int64 * 2)(0, 9), (ctypes.c_int64 * 1)(0))
    assert lib.dsa_workspace_size_varlen(ctypes.byref(ix), ctypes.byref(bad), 2048) == 256


def test_overlap_matrix_rejects_huge_k_without_overflow(lib):
    P = ctypes.c_void_p
    m = (ctypes.c_double * 4)()
    bufs = (P * 2)(FAKE, FAKE)
    for k in (2 ** 31 - 1, 2 ** 30, 60000):
        assert lib.topk_overlap_matrix(bufs, 2, 10, k, None, m, P(FAKE), 1 << 30, None) == UNSUPPORTED


# --- strides, size queries and the wait bound ---------------------------------------------

@pytest.mark.parametrize("field,value,status", [
    ("q_stride_t", 64 * 128 - 8, INVALID),   # tokens would overlap
    ("q_stride_t", 64 * 128 + 4, MISALIGNED),  # 8 bytes of bf16: not a multiple of 16
    ("q_stride_b", 4, MISALIGNED),
    ("k_stride_b", 12, MISALIGNED),
    ("q_stride_b", -16, INVALID),
    ("k_stride_b", -64, INVALID),
])
def test_indexer_stride_validation(lib, field, value, status):
    assert _topk_ix(lib, _ix(**{field: value})) == status


def test_indexer_strides_accepted_when_aligned(lib):
    # host validation passes; the call then fails only on the workspace it was not given
    ix = _ix(q_stride_t=64 * 128 + 64, q_stride_b=10 ** 7, k_stride_b=64 * 128 * 3)
    assert _topk_ix(lib, ix, ws_bytes=300) == WORKSPACE
    ix8 = _ix(dtype=dsa.DSA_E4M3, q_scale=FAKE, k_scale=FAKE, q_stride_t=64 * 128 + 16, k_stride_b=16)
    assert _topk_ix(lib, ix8, ws_bytes=300) == WORKSPACE
    ix8.q_stride_t = 64 * 128 + 8        # 8 bytes of e4m3 codes
    assert _topk_ix(lib, ix8, ws_bytes=300) == MISALIGNED


@pytest.mark.parametrize("field,value,status", [
    ("q_stride_t", 64 * 576 - 8, INVALID), ("q_stride_t", 64 * 576 + 4, MISALIGNED),
    ("q_stride_b", 12, MISALIGNED), ("k_stride_b", 6, MISALIGNED), ("v_stride_b", -8, INVALID),
])
def test_attention_stride_validation(lib, field, value, status):
    at = _at(**{field: value})
    r = lib.dsa_sparse_attn(ctypes.byref(at), ctypes.c_void_p(FAKE), 16, ctypes.c_void_p(FAKE), None,
                            ctypes.c_void_p(FAKE), 256, None)
    assert r == status


def test_topk_workspace_size_query(lib):
    # many rows: one CTA per row, no scratch beyond the flag word
    assert lib.dsa_topk_workspace_size(1, 4096, 131072, 0, 0, 2048) == 256
    # a few long rows: room for the split lists, a whole number of (k positions + k keys + count)
    # lists per row
    n = lib.dsa_topk_workspace_size(32, 1, 200000, 200000, 0, 2048)
    assert n > 256 and (n - 256) % (32 * (2048 * 8 + 4)) == 0
    # short rows are never split
    assert lib.dsa_topk_workspace_size(4, 1, 20000, 20000, 0, 2048) == 256
    # arguments the call would reject
    for args in ((0, 1, 10, 0, 0, 8), (1, 1, 10, 0, 2, 8), (1, 1, 10, -1, 0, 8), (1, 1, 10, 0, 0, 5000)):
        assert lib.dsa_topk_workspace_size(*args) == 256


def test_attention_workspace_size_query(lib):
    at = _at(B=32, T=1, S=200000)
    n = lib.dsa_attn_workspace_size(ctypes.byref(at), 2048)
    # split parts: fp32 outputs [64 x 512] and 64 LSEs per part, a whole number of parts per row
    assert n > 256 and (n - 256) % (32 * 64 * 513 * 4) == 0
    # enough rows: no split, one byte per row for the fixed-reference pass's row marks
    assert lib.dsa_attn_workspace_size(ctypes.byref(_at(B=1, T=4096)), 2048) == 256 + 4096
    assert lib.dsa_attn_workspace_size(ctypes.byref(_at(B=1, T=4000)), 2048) == 256 + 4096  # rounded to 256
    small = _at(H=8, d_qk=64, d_v=64, k_ld=64, v_ld=64, B=1, T=4)
    assert lib.dsa_attn_workspace_size(ctypes.byref(small), 64) == 256                # mma.sync shape
    assert lib.dsa_attn_workspace_size(None, 64) == 256
    # a short index row is not worth splitting: the row marks of its 32 rows
    assert lib.dsa_attn_workspace_size(ctypes.byref(at), 64) == 256 + 256


def test_group_workspace_size_covers_every_layer(lib):
    arr = (dsa.Layer * 4)()
    for i in range(4):
        arr[i].ix = _ix(B=32, T=1, S=200000, q_pos0=200000, dtype=dsa.DSA_E4M3, q_scale=FAKE, k_scale=FAKE)
        arr[i].at = _at(B=32, T=1, S=200000)
        arr[i].out = FAKE
    got = lib.indexshare_group_workspace_size(arr, 4, b"FSSS", 2048, None)
    want = max(lib.dsa_workspace_size(ctypes.byref(arr[0].ix), 2048),
               lib.dsa_attn_workspace_size(ctypes.byref(arr[0].at), 2048))
    assert got == want and got > 256
    assert lib.indexshare_group_workspace_size(arr, 4, b"FSS", 2048, None) == 256
    assert lib.indexshare_group_workspace_size(None, 4, b"FSSS", 2048, None) == 256
    # packed: the largest sequence's group need
    cu = [0, 1, 2]
    v = dsa.Varlen(2, (ctypes.c_int64 * 3)(*cu), (ctypes.c_int64 * 3)(0, 200000, 400000), (ctypes.c_int64 * 2)(200000, 200000))
    pk = (dsa.Layer * 4)()
    for i in range(4):
        pk[i].ix = _ix(B=1, T=2, S=400000, dtype=dsa.DSA_E4M3, q_scale=FAKE, k_scale=FAKE)
        pk[i].at = _at(B=1, T=2, S=400000)
        pk[i].out = FAKE
    one = (dsa.Layer * 4)()
    for i in range(4):
        one[i].ix = _ix(B=1, T=1, S=200000, q_pos0=200000, dtype=dsa.DSA_E4M3, q_scale=FAKE, k_scale=FAKE)
        one[i].at = _at(B=1, T=1, S=200000)
        one[i].out = FAKE
    assert lib.indexshare_group_workspace_size(pk, 4, b"FSSS", 2048, ctypes.byref(v)) == \
        lib.indexshare_group_workspace_size(one, 4, b"FSSS", 2048, None)


def test_wait_limit_setter_is_callable(lib):
    lib.dsa_set_wait_limit(100)
    lib.dsa_set_wait_limit(0)  # back to the default


def _draft(lib, ix, at, k=16, idx=FAKE, out=FAKE):
    return lib.indexshare_draft_forward(ctypes.byref(ix) if ix is not None else None, ctypes.byref(at), k,
                                        ctypes.c_void_p(idx) if idx else None,
                                        ctypes.c_void_p(out) if out else None, None, ctypes.c_void_p(FAKE), 256,
                                        None)


def test_draft_forward_validation(lib):
    ix, at = _ix(T=1), _at(T=4)
    assert _draft(lib, None, at) == INVALID
    assert _draft(lib, _ix(T=2), at) == INVALID      # the first step has one query per sequence
    assert _draft(lib, _ix(T=1, B=2), at) == INVALID  # sequences differ
    assert _draft(lib, _ix(T=1, S=32), at) == INVALID  # caches differ
    assert _draft(lib, ix, _at(T=4, H=32)) == UNSUPPORTED
    assert _draft(lib, ix, at, idx=0) == INVALID
    assert _draft(lib, ix, at, k=0) == UNSUPPORTED
    assert _draft(lib, ix, at, out=FAKE + 2) == MISALIGNED


def test_draft_workspace_size_covers_topk_and_attention(lib):
    ix = _ix(B=32, T=1, S=200000, q_pos0=200000, dtype=dsa.DSA_E4M3, q_scale=FAKE, k_scale=FAKE)
    at = _at(B=32, T=4, S=200000)
    n = lib.indexshare_draft_workspace_size(ctypes.byref(ix), ctypes.byref(at), 2048)
    assert n >= lib.dsa_workspace_size(ctypes.byref(ix), 2048)
    # the 128 draft rows fill the GPU without a decode split; one step alone splits its 32 rows
    assert n >= lib.dsa_attn_workspace_size(ctypes.byref(at), 2048)
    assert lib.indexshare_draft_workspace_size(None, ctypes.byref(at), 2048) == 256
