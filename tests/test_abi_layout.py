"""The ctypes mirrors of hsq_config and hsq_cache have the C layout of
include/hsq.h: a small C program compiled here with the system compiler
prints each field's offset and each struct's size, and the binding's
structures must match them field by field (no GPU needed)."""

import ctypes
import os
import shutil
import subprocess

import pytest

from hierarchical_kv_cache_hsq_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _c_layout(tmp_path, struct: str, fields):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / f"{struct}.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "hsq.h"', "int main(void) {",
             f'    printf("size %zu\\n", sizeof({struct}));']
    lines += [f'    printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ["    return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / struct
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}


@pytest.mark.parametrize("cls,struct", [(B.hsq_config, "hsq_config"), (B.hsq_cache, "hsq_cache")])
def test_ctypes_struct_matches_the_header(tmp_path, cls, struct):
    names = [f[0] for f in cls._fields_]
    c = _c_layout(tmp_path, struct, names)
    assert c["size"] == ctypes.sizeof(cls)
    for n in names:
        assert c[n] == getattr(cls, n).offset, n


def test_buffer_enum_matches_the_binding(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "bufs.c"
    names = [f"HSQ_BUF_{n.upper()}" for n in B.BUFFERS]
    body = "\n".join(f'    printf("%d\\n", (int){n});' for n in names)
    src.write_text('#include <stdio.h>\n#include "hsq.h"\nint main(void) {\n' + body +
                   '\n    printf("%d\\n", (int)HSQ_NBUF);\n    return 0;\n}\n')
    exe = tmp_path / "bufs"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert vals == list(range(len(B.BUFFERS))) + [B.HSQ_NBUF]
