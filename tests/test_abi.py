"""The C ABI library builds, loads and exports every entry point that
include/specverify.h declares; argument checks work without a GPU."""
import ctypes
import os
import re

import pytest

import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import build as svbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "specverify.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return sv.lib()


def test_header_declares_the_binding_symbols():
    assert _declared() == sorted(sv.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.spec_version() >= 1


def test_null_context_is_rejected_without_touching_a_gpu(lib):
    rc = lib.qgemm_w4a16(None, None, None, None, 64, None, None, 0, 16, 128, 64, None, 0, None)
    assert rc == -1
    assert b"null context" in lib.spec_last_error()
    assert lib.spec_destroy(None) == 0


def test_create_out_pointer_checked(lib):
    assert lib.spec_create(0, 0, None) == -1


def _declared_params():
    """(name, [parameter declarations]) for every function in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
        params = [p.strip() for p in m.group(2).replace("\n", " ").split(",")]
        out[m.group(1)] = [p for p in params if p and p != "void"]
    return out


def _kind_of_param(decl: str) -> str:
    if "*" in decl:
        return "pointer"
    if decl.startswith(("uint64_t", "size_t")):
        return "u64"
    if decl.startswith("int"):
        return "i32"
    raise AssertionError(f"unexpected parameter type: {decl}")


def _kind_of_ctype(t) -> str:
    if t is ctypes.c_void_p or issubclass(t, ctypes._Pointer):
        return "pointer"
    if ctypes.sizeof(t) == 8:
        return "u64"
    if ctypes.sizeof(t) == 4:
        return "i32"
    raise AssertionError(f"unexpected ctype: {t}")


def test_binding_argument_lists_match_the_header():
    # a missing or mistyped argument would pass garbage through the C ABI
    decl = _declared_params()
    for name, argtypes in sv._SIGS.items():
        want = [_kind_of_param(p) for p in decl[name]]
        got = [_kind_of_ctype(t) for t in argtypes]
        assert got == want, (name, got, want)


def _struct_fields(name):
    """[(field type, field name)] of a typedef'd struct in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct " + name + r"\s*\{(.*?)\}", text, flags=re.S).group(1)
    out = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        m = re.match(r"(.*?)(\w+(?:\s*,\s*\w+)*)$", decl)
        ty, names = m.group(1).strip(), m.group(2)
        for n in names.split(","):
            out.append((ty, n.strip()))
    return out


def test_gemm_desc_layout_matches_the_header():
    # the stack descriptor crosses the ABI as an array of structs: same fields,
    # same order, same kinds
    fields = _struct_fields("spec_gemm_desc")
    assert [n for _, n in fields] == [n for n, _ in sv.GemmDesc._fields_]
    for (ty, n), (_, ct) in zip(fields, sv.GemmDesc._fields_):
        assert _kind_of_param(ty + (" *" if "*" in ty else "")) == _kind_of_ctype(ct), n
