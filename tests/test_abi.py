"""The C-ABI library loads on the CPU host and exports every entry point bskv.h declares."""

import ctypes
import os
import re

import block_sparse_kv_gb300 as bskv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "bskv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bskv_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    so = ctypes.CDLL(bskv.build.LIB if hasattr(bskv.build, "LIB") else bskv._build.LIB)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing


def test_binding_covers_the_abi(lib):
    for n in _declared():
        assert n in bskv._SIGS, n


def test_version_and_error_text(lib):
    assert bskv.bskv_version() >= 100
    try:
        bskv.bskv_plan_mla_sparse([8], 1, 1, 4, 100, num_sms=4)
    except bskv.BskvError as e:
        assert e.status == "ERR_INVALID_ARG"
        assert "divisible by 64" in str(e)
    else:
        raise AssertionError("top_k % 64 != 0 accepted")


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "block_sparse_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("the oracle", ""), f
