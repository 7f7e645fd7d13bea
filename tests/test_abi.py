"""The C ABI library: it builds, loads, and exports every entry point the header declares (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coli_moe.h")


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^COLI_API\s+[\w\s\*]+?\b(coli_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    from int4_grouped_expert_router_gb300.build import build
    path = build()
    return ctypes.CDLL(path), path


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ("coli_init", "coli_destroy", "coli_router_select", "coli_expert_upload", "coli_expert_free",
                 "coli_expert_table_set", "coli_expert_group", "coli_check_error", "coli_last_error"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    cdll, path = lib
    for name in header_functions():
        assert hasattr(cdll, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    assert set(header_functions()) <= exported
    # nothing but the C ABI leaks out of the library
    assert {s for s in exported if s.startswith("coli")} == set(header_functions())


def test_binding_matches_header():
    from int4_grouped_expert_router_gb300 import binding as B
    assert set(B.SIGNATURES) == set(header_functions())


def test_init_without_a_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cdll, _ = lib
    out = ctypes.c_void_p(123)
    rc = cdll.coli_init(ctypes.byref(out), 0, None)
    assert rc == -3 and out.value is None   # COLI_E_CUDA, *out cleared


def test_null_context_is_rejected(lib):
    cdll, _ = lib
    cdll.coli_check_error.restype = ctypes.c_int
    assert cdll.coli_check_error(None) == -1
    cdll.coli_expert_upload.restype = ctypes.c_uint64
    assert cdll.coli_expert_upload(None, None, None, 1, 2, 0) == 0
