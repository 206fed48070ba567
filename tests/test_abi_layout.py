"""The ctypes structures of the Python binding have the layout of the C ABI's
structures: a small C program compiled against include/dsa.h prints every
field's offset and each structure's size, and the binding must agree (a
mismatch would hand the library shifted fields). Needs only gcc."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

from deepseek_v4_sparse_ratio_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = {"dsa_pool_state": B.dsa_pool_state, "dsa_prefill_workspace": B.dsa_prefill_workspace}


def _c_layout():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "dsa.h"', "int main(void) {"]
    for name, cls in STRUCTS.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(src, "w") as fh:
            fh.write("\n".join(lines) + "\n")
        subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    layout = {}
    for line in out.splitlines():
        name, field, value = line.split()
        layout[(name, field)] = int(value)
    return layout


def test_binding_structs_match_the_c_header():
    layout = _c_layout()
    for name, cls in STRUCTS.items():
        assert ctypes.sizeof(cls) == layout[(name, "size")], name
        for field, _ in cls._fields_:
            assert getattr(cls, field).offset == layout[(name, field)], (name, field)


def _prototypes():
    """name -> parameter count, from the prototypes in include/dsa.h."""
    import re
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(?:int|size_t|const char \*)\s*(dsa_\w+)\s*\(([^;{]*?)\)\s*;", text):
        params = [p for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        protos[m.group(1)] = len(params)
    return protos


def test_binding_argtypes_match_the_prototypes():
    protos = _prototypes()
    lib = B.load()
    for name in B.EXPORTS:
        assert name in protos, name
        argtypes = getattr(lib, name).argtypes
        if argtypes is not None:
            assert len(argtypes) == protos[name], (name, len(argtypes), protos[name])


def test_binding_error_codes_match_the_header():
    import re
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(DSA_\w+)\s*=\s*(-?\d+)", text)}
    errs = {k: v for k, v in codes.items() if k.startswith("DSA_ERR_") or k == "DSA_OK"}
    assert len(errs) >= 11
    for name, value in errs.items():
        if hasattr(B, name):
            assert getattr(B, name) == value, name
    assert all(hasattr(B, n) for n in errs if n != "DSA_OK"), "an error code is missing"


def test_static_scratch_size_matches_the_header():
    import re
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    m = re.search(r"#define\s+DSA_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m is not None
    assert B.DSA_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
