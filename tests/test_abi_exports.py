"""The C-ABI library loads and exports every function include/*.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s+\**([A-Za-z_]\w*)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from resident_brute_force_gb300 import _build
    _build.build()
    return ctypes.CDLL(_build.LIB_PATH)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("upload_corpus_rowmajor", "search_resident", "search_resident_batch", "topk_int32",
                     "rbf_create", "rbf_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_covers_the_header():
    from resident_brute_force_gb300 import SIGNATURES
    assert sorted(SIGNATURES) == declared_functions()


def test_status_strings_without_gpu(lib):
    lib.rbf_status_string.restype = ctypes.c_char_p
    assert lib.rbf_status_string(0) == b"RBF_OK"
    assert lib.rbf_status_string(5) == b"RBF_ERR_TIMEOUT"


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "resident_brute_force_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                for bad in ("import oracle", "from oracle", "liboracle", "oracle.c"):
                    assert bad not in text, (f, bad)


def test_checked_build_exports_the_same_boundary():
    """The checked build (-DRBF_CHECKS) compiles, exports every declared
    function and names its extra status."""
    from resident_brute_force_gb300 import _build
    checked = ctypes.CDLL(_build.build(checks=True))
    for name in declared_functions():
        assert hasattr(checked, name), name
    checked.rbf_status_string.restype = ctypes.c_char_p
    assert checked.rbf_status_string(7) == b"RBF_ERR_BOUNDS"
