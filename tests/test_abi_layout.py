"""The ctypes binding's structs lay out like include/skv.h's (no GPU needed).

A C program built from the header with the host C compiler prints every field's offset
and every struct's size; the binding's ctypes classes must match them field by field,
so a field added to the header and not to the binding (or in another order) fails here
instead of being read past the end of a Python-made struct.
"""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from top_sparse_kv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = {
    "skv_problem": binding.CProblem,
    "skv_kv_pool": binding.CPool,
    "skv_index_src": binding.CIndex,
    "skv_prefetch": binding.CPrefetch,
    "skv_slot_cache": binding.CSlotCache,
    "skv_paris": binding.CParis,
    "skv_paris_index": binding.CParisIndex,
}


def _c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "skv.h"', "int main(void) {"]
    for cname, cls in STRUCTS.items():
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    layout = {}
    for line in out.splitlines():
        struct, field, value = line.split()
        layout[(struct, field)] = int(value)
    return layout


def test_binding_structs_match_the_header(tmp_path):
    layout = _c_layout(tmp_path)
    for cname, cls in STRUCTS.items():
        assert ctypes.sizeof(cls) == layout[(cname, "sizeof")], cname
        for fname, _ in cls._fields_:
            assert getattr(cls, fname).offset == layout[(cname, fname)], (cname, fname)


def test_every_header_struct_field_is_in_the_binding():
    # the header's field names, in order, against the binding's (a field the binding
    # lacks would not be caught by the offsets of the fields it has)
    text = re.sub(r"/\*.*?\*/", " ", open(os.path.join(ROOT, "include", "skv.h")).read(), flags=re.S)
    for cname, cls in STRUCTS.items():
        body = text.split(f"typedef struct {cname} {{", 1)[1].split("}", 1)[0]
        names = [d.replace("*", " ").split()[-1] for d in body.split(";") if d.strip()]
        assert names == [f for f, _ in cls._fields_], cname
