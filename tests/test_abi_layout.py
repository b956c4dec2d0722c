"""The ctypes argument structs of the Python binding mirror include/nvfp4.h
field for field: the same names in the same order at the same byte offsets,
and the same struct sizes.  A small C program built with the host compiler
prints offsetof/sizeof for every field; nothing runs on a device."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from nvfp4_block_scaled_06_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MIRRORS = {
    "nvfp4_quant_args": B.QuantArgs,
    "nvfp4_gemm_args": B.GemmArgs,
    "nvfp4_grouped_args": B.GroupedArgs,
    "nvfp4_lora_args": B.LoraArgs,
    "nvfp4_dequant_args": B.DequantArgs,
    "nvfp4_dgrad_args": B.DgradArgs,
    "nvfp4_wgrad_args": B.WgradArgs,
    "nvfp4_moe_down_args": B.MoeDownArgs,
}


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    d = tmp_path_factory.mktemp("abi")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "nvfp4.h"', "int main(void) {"]
    for cname, cls in MIRRORS.items():
        lines.append(f'  printf("{cname} . %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = d / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = d / "layout"
    # a field the header lacks fails to compile: the message names it
    r = subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    table = {}
    for ln in out.splitlines():
        cname, fname, val = ln.split()
        table[(cname, fname)] = int(val)
    return table


def header_fields(cname):
    """Field names of a typedef'd struct in the header, in declaration order."""
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    m = re.search(r"typedef struct\s*\{([^{}]*)\}\s*" + cname + r"\s*;", src)
    assert m, cname
    names = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "const float *a, *b" -> a, b
        for part in decl.split(","):
            names.append(re.findall(r"[A-Za-z_][A-Za-z0-9_]*", part)[-1])
    return names


@pytest.mark.parametrize("cname", sorted(MIRRORS))
def test_struct_mirrors_header(cname, c_layout):
    cls = MIRRORS[cname]
    assert [f for f, _ in cls._fields_] == header_fields(cname)
    for fname, _ in cls._fields_:
        assert getattr(cls, fname).offset == c_layout[(cname, fname)], fname
    assert ctypes.sizeof(cls) == c_layout[(cname, ".")]
