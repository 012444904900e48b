"""The checked library (built with GBATTN_CHECKED=1, selected at load time by the
environment variable GBATTN_CHECKED=1) without a GPU: it builds beside the plain
one, exports the same symbols, says it is the checked build, and its extent
arithmetic -- the test every device-computed index passes before an access --
gives the right answer on the edges of fixed-length and packed tensors."""

import ctypes
import os
import shutil
import subprocess

import pytest

from bwd_flashattention_fwd_sm_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_library_exports_every_symbol():
    build.build()
    assert os.path.exists(build.LIB_CHECKED)
    lib = ctypes.CDLL(build.LIB_CHECKED)
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    assert lib.attn_version().endswith(b" checked")
    plain = ctypes.CDLL(build.LIB)
    plain.attn_version.restype = ctypes.c_char_p
    assert not plain.attn_version().endswith(b" checked")


def test_environment_selects_the_checked_library(monkeypatch):
    monkeypatch.setenv("GBATTN_CHECKED", "1")
    assert _lib.library_path() == build.LIB_CHECKED
    monkeypatch.setenv("GBATTN_CHECKED", "0")
    assert _lib.library_path() == build.LIB


def test_extent_arithmetic_on_the_host(tmp_path):
    nvcc = build.nvcc()
    if not shutil.which(nvcc) and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "extents")
    src = os.path.join(ROOT, "tests", "checked_extents_host.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-I", build.CSRC, "-I", build.INCLUDE, src, "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout
