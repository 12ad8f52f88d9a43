"""The Python binding's ctypes structures against the C header, on the CPU:
a small C program built against include/fdl.h with the host compiler prints
every struct's size and each field's offset, and those must equal the ctypes
layout field by field (names in the same order, same offsets, same size)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import kv_cache_attention_gb300 as fdl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = ("fdl_config", "fdl_unmask_args", "fdl_model", "fdl_refresh_args", "fdl_flash_params", "fdl_flash_seqs",
           "fdl_flash_trace")


def _c_fields(name: str, header: str):
    """Field names of ``typedef struct { ... } name;`` in declaration order."""
    end = re.search(r"\}\s*" + name + r"\s*;", header)
    assert end, name
    start = header.rfind("typedef struct {", 0, end.start())
    body = re.sub(r"/\*.*?\*/", "", header[start + len("typedef struct {"):end.start()], flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "int* a; int b, c" style: the declarators after the type
        parts = re.split(r",", decl)
        first = re.findall(r"([A-Za-z_][A-Za-z0-9_]*)\s*$", parts[0])
        names.append(first[0])
        for p in parts[1:]:
            names.append(re.findall(r"([A-Za-z_][A-Za-z0-9_]*)\s*$", p.strip())[0])
    return names


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    header = open(os.path.join(ROOT, "include", "fdl.h")).read()
    fields = {s: _c_fields(s, header) for s in STRUCTS}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fdl.h"', "int main(void) {"]
    for s, names in fields.items():
        lines.append(f'  printf("{s} size %zu\\n", sizeof({s}));')
        for n in names:
            lines.append(f'  printf("{s} {n} %zu\\n", offsetof({s}, {n}));')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    layout = {}
    for line in out:
        if line.strip():
            s, f, v = line.split()
            layout.setdefault(s, {})[f] = int(v)
    return fields, layout


@pytest.mark.parametrize("name", STRUCTS)
def test_binding_struct_matches_the_header(c_layout, name):
    fields, layout = c_layout
    py = getattr(fdl, name)
    assert [f[0] for f in py._fields_] == fields[name]
    assert ctypes.sizeof(py) == layout[name]["size"], name
    for f in fields[name]:
        assert getattr(py, f).offset == layout[name][f], (name, f)
