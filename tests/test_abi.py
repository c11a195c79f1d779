"""The C ABI library loads on a machine without a GPU, exports every entry point that
include/csa2.h declares, and rejects invalid calls on the host before any launch."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")
LIB = os.path.join(ROOT, "sparse_attention_csa2_gb300", "_lib", "libcsa2.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        subprocess.run([sys.executable, os.path.join(ROOT, "sparse_attention_csa2_gb300", "_build.py")], check=True)
    return ctypes.CDLL(LIB)


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z0-9_]+\s*\*?\s*(csa2_[a-z0-9_]+)\s*\(", src, re.M)))


def test_header_declares_the_five_calls():
    names = declared()
    for n in ("csa2_index_scores", "csa2_block_pool", "csa2_topk", "csa2_sparse_attn", "csa2_fused_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(1) == b"invalid argument"
    assert lib.csa2_version() == 0x000100


def test_invalid_calls_are_rejected_on_the_host(lib):
    # NULL argument structs: rejected before anything touches CUDA
    for n in ("csa2_index_scores", "csa2_topk", "csa2_block_pool", "csa2_sparse_attn", "csa2_fused_decode"):
        f = getattr(lib, n)
        f.restype = ctypes.c_int
        assert f(None, None) == 1, n
    lib.csa2_read_device_status.restype = ctypes.c_int
    assert lib.csa2_read_device_status(None, None, None) == 1


def test_next_row_calls_reject_invalid_arguments_on_the_host(lib):
    """The writer, compressor, expansion and projection entry points validate shapes, pointers
    and alignment before any launch (no GPU needed to reach these answers)."""
    for n in ("csa2_write_records", "csa2_compress", "csa2_expand_mxfp4", "csa2_linear", "csa2_query_proj",
              "csa2_out_proj"):
        f = getattr(lib, n)
        f.restype = ctypes.c_int
        assert f(None, None) == 1, n

    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

    class Linear(ctypes.Structure):
        _fields_ = [("n_tokens", i32), ("in_features", i32), ("out_features", i32), ("x", vp), ("w", vp),
                    ("out", vp), ("dev_status", vp)]

    class QueryProj(ctypes.Structure):
        _fields_ = [("n_tokens", i32), ("hidden", i32), ("q_rank", i32), ("n_heads", i32), ("x", vp), ("w_dq", vp),
                    ("g_q", vp), ("w_uq", vp), ("g_head", vp), ("eps", f32), ("q", vp), ("workspace", vp),
                    ("workspace_bytes", sz), ("dev_status", vp)]

    class OutProj(ctypes.Structure):
        _fields_ = [("n_tokens", i32), ("n_heads", i32), ("n_groups", i32), ("o_rank", i32), ("hidden", i32),
                    ("o", vp), ("w_oa", vp), ("w_ob", vp), ("out", vp), ("workspace", vp), ("workspace_bytes", sz),
                    ("dev_status", vp)]

    class Expand(ctypes.Structure):
        _fields_ = [("n_records", i64), ("codes", vp), ("exps", vp), ("out", vp)]

    A = 1 << 20  # a 16-byte-aligned stand-in address: never dereferenced, every case fails validation first
    lin = lib.csa2_linear
    assert lin(ctypes.byref(Linear(0, 64, 128, None, None, None, None)), None) == 0   # nothing to do
    assert lin(ctypes.byref(Linear(4, 65, 128, A, A, A, None)), None) == 1            # K not a multiple of 64
    assert lin(ctypes.byref(Linear(4, 64, 100, A, A, A, None)), None) == 1            # features not of 128
    assert lin(ctypes.byref(Linear(4, 64, 128, A + 8, A, A, None)), None) == 1        # misaligned x
    assert lin(ctypes.byref(Linear(-1, 64, 128, A, A, A, None)), None) == 1

    qp = lib.csa2_query_proj
    qp_ws = lib.csa2_query_proj_workspace_size
    qp_ws.restype = sz
    good = QueryProj(32, 4096, 1024, 64, A, A, None, A, None, 1e-6, A, A, 0, None)
    need = qp_ws(ctypes.byref(good))
    assert need == (32 * 1024 * 2 + 255) // 256 * 256 + (8 * 8 * 32 * 4 + 255) // 256 * 256
    assert qp(ctypes.byref(good), None) == 5                                          # workspace too small
    for field, bad in (("q_rank", 1000), ("hidden", 100), ("n_heads", 0), ("eps", -1.0)):
        a = QueryProj(32, 4096, 1024, 64, A, A, None, A, None, 1e-6, A, A, need, None)
        setattr(a, field, bad)
        assert qp(ctypes.byref(a), None) == 1, field

    op = lib.csa2_out_proj
    for args in ((4, 64, 7, 1024, 4096), (4, 64, 8, 1000, 4096), (4, 64, 8, 1024, 4000), (4, 4, 8, 1024, 4096)):
        assert op(ctypes.byref(OutProj(*args, A, A, A, A, A, 1 << 30, None)), None) == 1, args
    assert op(ctypes.byref(OutProj(4, 64, 8, 1024, 4096, A, A, A, A, None, 0, None)), None) == 5

    ex = lib.csa2_expand_mxfp4
    assert ex(ctypes.byref(Expand(0, None, None, None)), None) == 0
    assert ex(ctypes.byref(Expand(10, A + 4, A, A)), None) == 1                       # misaligned codes
    assert ex(ctypes.byref(Expand(10, A, None, A)), None) == 1


class _TopkArgs(ctypes.Structure):
    _fields_ = [("scores", ctypes.c_void_p), ("cand", ctypes.c_void_p), ("n_valid", ctypes.c_void_p),
                ("n_rows", ctypes.c_int32), ("L", ctypes.c_int64), ("K", ctypes.c_int32), ("idx", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


@pytest.mark.parametrize("name", ["csa2_topk", "csa2_topk_static"])
def test_topk_entry_points_validate_on_the_host(lib, name):
    """Both top-K entry points reject the same invalid requests before touching CUDA: a NULL
    argument struct, NULL scores / n_valid / idx, L outside 1 .. 2^24 (EINVAL), K outside
    1 .. CSA2_MAX_TOPK (EUNSUPPORTED); zero rows is a valid call that does nothing."""
    f = getattr(lib, name)
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_TopkArgs), ctypes.c_void_p]
    assert f(None, None) == 1
    A = 1 << 20  # an aligned stand-in address: every case below fails validation before any use

    def call(**kw):
        a = _TopkArgs(A, None, A, 4, 1000, 64, A, None, 0)
        for k, v in kw.items():
            setattr(a, k, v)
        return f(ctypes.byref(a), None)

    assert call(n_rows=0) == 0
    assert call(n_rows=-1) == 1
    assert call(scores=None) == 1
    assert call(n_valid=None) == 1
    assert call(idx=None) == 1
    assert call(L=0) == 1
    assert call(L=(1 << 24) + 1) == 1
    assert call(K=0) == 2
    assert call(K=1025) == 2


def test_tuning_overrides_are_range_checked(lib):
    st = lib.csa2_set_tuning
    st.restype = ctypes.c_int
    st.argtypes = [ctypes.c_int32, ctypes.c_int32]
    assert st(-1, 0) == 1 and st(5, 0) == 1            # unknown knobs
    assert st(0, 65) == 1 and st(0, -1) == 1           # scan segments 0..64
    assert st(3, 9) == 1                               # projection K split 0..8
    assert st(0, 8) == 0 and st(0, 0) == 0             # set, and back to automatic
    assert st(2, 0) == 0 and st(2, 1) == 0
    assert st(4, 5) == 1 and st(4, -1) == 1           # attention kernel 0..4
    assert st(4, 4) == 0 and st(4, 0) == 0
