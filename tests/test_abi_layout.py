"""The binding's ctypes structs have the C header's layout: a small C program,
compiled here against include/kpool_dsa.h, prints sizeof and offsetof of
every field of every struct the binding mirrors, and each must equal the
ctypes figure (a field added, dropped, reordered or retyped on one side only
fails here, before any call reaches the library)."""
import ctypes
import os
import subprocess

import pytest

import dsa_indexer_sparse_kpool_b300 as kp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = [name for name in dir(kp) if name.startswith("kp_")
           and isinstance(getattr(kp, name), type) and issubclass(getattr(kp, name), ctypes.Structure)]


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kpool_dsa.h"', "int main(void) {"]
    for name in STRUCTS:
        lines.append(f'    printf("{name} sizeof %zu\\n", sizeof({name}));')
        for field, _ in getattr(kp, name)._fields_:
            lines.append(f'    printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["    return 0;", "}"]
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {tuple(l.split()[:2]): int(l.split()[2]) for l in out.splitlines()}


def test_every_struct_is_mirrored():
    header = open(os.path.join(ROOT, "include", "kpool_dsa.h")).read()
    declared = {l.split()[2] for l in header.splitlines() if l.startswith("typedef struct kp_")}
    assert declared == set(STRUCTS)


@pytest.mark.parametrize("name", STRUCTS)
def test_struct_layout_matches_the_header(c_layout, name):
    cls = getattr(kp, name)
    assert c_layout[(name, "sizeof")] == ctypes.sizeof(cls)
    for field, _ in cls._fields_:
        assert c_layout[(name, field)] == getattr(cls, field).offset, field
