"""The C-ABI library builds, loads without a GPU and exports every entry
point include/wedlm.h declares; the ctypes mirrors of its structs have the
sizes and field offsets gcc computes from the header."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wedlm.h")


@pytest.fixture(scope="module")
def lib():
    from serving_wedlm_step_gb300.build import build
    build()
    from serving_wedlm_step_gb300 import binding
    return binding.load_library()


def declared_functions():
    names = []
    for path in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not path.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", path)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(wedlm_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_step_boundary():
    names = declared_functions()
    for n in ("wedlm_create", "wedlm_step", "wedlm_get_status", "wedlm_last_error",
              "wedlm_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (wedlm_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_lists_every_export():
    from serving_wedlm_step_gb300 import binding
    assert sorted(binding.EXPORTED) == declared_functions()


def test_ctypes_struct_layout_matches_c():
    from serving_wedlm_step_gb300 import binding as b
    structs = {"wedlm_config": b.Config, "wedlm_weights": b.Weights,
               "wedlm_slot_rec": b.SlotRec, "wedlm_step_in": b.StepIn,
               "wedlm_step_out": b.StepOut, "wedlm_gen_in": b.GenIn}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', 'int main(void){']
    for cname, py in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname}.{fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0;}")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(src, "w").write("\n".join(lines))
        subprocess.run(["gcc", "-std=c99", "-o", exe, src], check=True)
        got = dict(l.split() for l in subprocess.run([exe], capture_output=True, text=True,
                                                      check=True).stdout.splitlines())
    for cname, py in structs.items():
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert int(got[f"{cname}.{fname}"]) == getattr(py, fname).offset, (cname, fname)


def test_constants_match_header():
    from serving_wedlm_step_gb300 import binding as b
    text = open(HEADER).read()
    assert re.search(r"WEDLM_KIND_COUNT", text)
    kinds = re.search(r"WEDLM_KIND_REORDER = 0,(.*?)WEDLM_KIND_COUNT", text, re.S).group(1)
    n_kinds = 1 + len(re.findall(r"WEDLM_KIND_\w+", kinds))
    assert n_kinds == len(b.KINDS)
    for name, val in (("WEDLM_DEV_BAD_PAGE", b.DEV_BAD_PAGE), ("WEDLM_DEV_CAPACITY", b.DEV_CAPACITY),
                      ("WEDLM_DEV_BAD_TOKEN", b.DEV_BAD_TOKEN), ("WEDLM_DEV_NUMERIC", b.DEV_NUMERIC),
                      ("WEDLM_DEV_TIMEOUT", b.DEV_TIMEOUT), ("WEDLM_DEV_BAD_SEQLEN", b.DEV_BAD_SEQLEN)):
        assert re.search(rf"{name} = {val}\b", text), name
