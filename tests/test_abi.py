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
