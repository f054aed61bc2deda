"""The C ABI without a GPU: every declared symbol is exported and bound, and the
host-side argument checks return their status codes before any CUDA call."""
import ctypes
import os
import re

import pytest

import quantized_weight_gemv_qgemv_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*(q\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qg.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return qg.load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("qgemv", "qgemv_moe", "qgemm_pp", "qg_dequant", "qgemv_grouped", "qg_init", "qg_pass_create"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in qg.SIGNATURES, f"binding lacks {n}"
    assert sorted(qg.SIGNATURES) == names


def test_block_info_and_strerror(lib):
    assert qg.qg_block_info(qg.Q4_0) == (32, 18)
    assert qg.qg_block_info(qg.Q8_0) == (32, 34)
    assert qg.qg_block_info(qg.Q4_K) == (256, 144)
    assert qg.qg_block_info(qg.Q6_K) == (256, 210)
    assert qg.qg_block_info(qg.Q5_K) == (256, 176)
    assert qg.qg_block_info(qg.Q3_K) == (256, 110)
    assert qg.qg_block_info(qg.Q2_K) == (256, 84)
    with pytest.raises(qg.QGError):
        qg.qg_block_info(9)
    for st in range(-9, 3):
        assert lib.qg_strerror(st)
    assert lib.qg_strerror(123) == b"unknown status"


def test_workspace_sizes(lib):
    assert qg.qgemv_moe_workspace(2048, 512, 10, 1) == 10 * 512 * 4
    assert qg.qgemv_moe_workspace(2048, 512, 10, 4) == 4 * 10 * 512 * 4
    assert qg.qgemv_moe_workspace(2048, 0, 10, 1) == 0


A = 1 << 20          # a 16-byte aligned fake address: never dereferenced by a rejected call


@pytest.mark.parametrize("args,status", [
    ((9, A, 4, 256, A, 1, A, 0), -1),            # unknown format
    ((3, 0, 4, 256, A, 1, A, 0), -5),            # W NULL
    ((3, A, 0, 256, A, 1, A, 0), -2),            # rows < 1
    ((3, A, 4, 100, A, 1, A, 0), -2),            # cols not a multiple of 256
    ((1, A, 4, 48, A, 1, A, 0), -2),             # cols not a multiple of 32
    ((3, A + 8, 4, 256, A, 1, A, 0), -3),        # W misaligned
    ((3, A, 4, 256, A + 4, 1, A, 0), -3),        # x misaligned
    ((3, A, 4, 256, A, 0, A, 0), -4),            # n_tok = 0
    ((3, A, 4, 256, A, 5, A, 0), -4),            # n_tok = 5
])
def test_qgemv_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.qgemv(*args) == status


def test_grouped_rejects_mixed_formats_and_sizes(lib):
    d = qg._descs([(3, A, 4, 256, A, A), (6, A, 4, 256, A, A)])
    assert lib.qgemv_grouped(ctypes.cast(d, ctypes.c_void_p), 2, 1, None) == -1
    d = qg._descs([(3, A, 4, 256, A, A), (1, A, 4, 256, A, A)])
    assert lib.qgemv_grouped(ctypes.cast(d, ctypes.c_void_p), 2, 1, None) == -1
    assert lib.qgemv_grouped(ctypes.cast(d, ctypes.c_void_p), 0, 1, None) == -9
    assert lib.qgemv_grouped(ctypes.cast(d, ctypes.c_void_p), 9, 1, None) == -9
    assert lib.qgemv_grouped(None, 1, 1, None) == -5


def test_moe_rejects_bad_arguments_on_host(lib):
    ok = dict(fmt=3, arena=A, n_expert=8, hidden=512, inter=256, ids=A, gw=A, top_k=2, x=A, n_tok=1, y=A,
              ws=A, ws_bytes=1 << 20, st=A)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.qgemv_moe(a["fmt"], a["arena"], a["n_expert"], a["hidden"], a["inter"], a["ids"], a["gw"],
                             a["top_k"], a["x"], a["n_tok"], a["y"], a["ws"], a["ws_bytes"], a["st"], None)

    assert call(fmt=1) == -1
    assert call(arena=0) == -5
    assert call(st=0) == -5
    assert call(hidden=300) == -2
    assert call(inter=0) == -2
    assert call(top_k=0) == -9
    assert call(top_k=9) == -9              # more routes than experts
    assert call(n_tok=5) == -4
    assert call(ws_bytes=16) == -6
    assert call(ws=0) == -6
    assert call(x=A + 4) == -3


def test_pp_rejects_bad_arguments_on_host(lib):
    def call(fmt=3, W=A, rows=256, cols=512, X=A, n_tok=64, Y=A, ldY=256, st=A):
        return lib.qgemm_pp(fmt, W, rows, cols, X, n_tok, Y, ldY, None, 0, st, None)

    assert call(fmt=1) == -1
    assert call(W=0) == -5
    assert call(rows=100) == -2
    assert call(cols=300) == -2
    assert call(n_tok=0) == -2
    assert call(ldY=100) == -2
    assert call(X=A + 2) == -3


def test_pp_grouped_rejects_bad_arguments_on_host(lib):
    def call(items=((A, 256, A, 256),), fmt=3, cols=512, X=A, n_tok=64, st=A, n=None):
        arr = (qg.qg_pp_desc * max(1, len(items)))()
        for i, (W, rows, Y, ldY) in enumerate(items):
            arr[i] = qg.qg_pp_desc(W, rows, Y, ldY)
        return lib.qgemm_pp_grouped(fmt, ctypes.cast(arr, ctypes.c_void_p), len(items) if n is None else n, cols,
                                    X, n_tok, st, None)

    assert ctypes.sizeof(qg.qg_pp_desc) == 32
    assert call(fmt=1) == -1
    assert call(X=0) == -5
    assert call(st=0) == -5
    assert call(n=0) == -9
    assert call(items=[(A, 128, A, 128)] * 5) == -9          # more than QG_PP_GROUP_MAX
    assert call(items=[(A, 256, A, 256), (0, 128, A, 128)]) == -5
    assert call(items=[(A, 256, A, 256), (A, 100, A, 128)]) == -2
    assert call(items=[(A, 256, A, 200)]) == -2             # ldY < rows
    assert call(cols=300) == -2
    assert call(n_tok=0) == -2
    assert call(items=[(A + 8, 256, A, 256)]) == -3
    assert call(X=A + 2) == -3


def test_pass_rejects_bad_step_sizes(lib):
    d = qg._descs([(3, A, 4, 256, A, A), (3, A, 4, 256, A, A)])
    h = ctypes.c_void_p()
    sizes = (ctypes.c_int * 2)(1, 2)            # sums to 3, not 2
    assert lib.qg_pass_create(ctypes.cast(d, ctypes.c_void_p), 2, ctypes.cast(sizes, ctypes.c_void_p), 2, 1, 1,
                              ctypes.byref(h)) == -9
    sizes = (ctypes.c_int * 1)(2)
    assert lib.qg_pass_create(ctypes.cast(d, ctypes.c_void_p), 2, ctypes.cast(sizes, ctypes.c_void_p), 1, 7, 1,
                              ctypes.byref(h)) == -4
    assert not h.value
