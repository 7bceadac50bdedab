"""libtopk loads, exports every declared entry point, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

import sparse_attention_row_gb300 as sar
from sparse_attention_row_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return ctypes.CDLL(sar.library_path())


def declared_functions():
    text = open(os.path.join(ROOT, "include", "libtopk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(topk_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(sar.EXPORTED) == set(names), names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(0, 9):
        assert sar.topk_status_string(code)
    assert sar.topk_status_string(2).startswith("topk must be")


def test_host_validation_needs_no_gpu(lib):
    fake = 0x10000  # never dereferenced: validation fails before any CUDA call
    assert sar.topk_ragged(fake, 4096, fake, 8, 1, 0, fake, fake, None) == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert sar.topk_ragged(fake, 4096, fake, 8, 1, 4097, fake, fake, None) == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert sar.topk_ragged_static(fake, 4096, fake, 8, 1, -5, fake, None) == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert sar.topk_ragged(fake, 4096, fake, -1, 1, 512, fake, fake, None) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged(fake, 0, fake, 8, 1, 512, fake, fake, None) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged(fake, 4096, fake, 9, 2, 512, fake, fake, None) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged(fake, 4096, fake, 0, 1, 512, fake, fake, None) == sar.TOPK_OK
    assert sar.topk_ragged(None, 4096, fake, 8, 1, 512, fake, fake, None) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged(fake + 2, 4096, fake, 8, 1, 512, fake, fake, None) == sar.TOPK_ERR_MISALIGNED
    assert sar.topk_ragged(fake, 4096, fake, 8, 1, 512, fake, fake + 4, None) == sar.TOPK_ERR_MISALIGNED
    assert sar.topk_workspace_init(None, 1024, None) == sar.TOPK_ERR_INVALID_ARG
    # strided views: column stride and column count are checked before anything else
    assert sar.topk_ragged_strided(fake, 4096, 0, 4096, fake, 8, 1, 512, fake, fake) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged_strided(fake, 4096, 2, 0, fake, 8, 1, 512, fake, fake) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged_strided(fake, -1, 2, 100, fake, 8, 1, 512, fake, fake) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_ragged_strided(fake, 1, 8, 100, fake, 8, 1, 0, fake, fake) == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert sar.topk_ragged_strided(fake, 1, 8, 100, fake, 0, 1, 512, fake, fake) == sar.TOPK_OK
    # values and order of selected rows
    assert sar.topk_gather_sort(fake, 100, 0, 100, 8, 512, fake) == sar.TOPK_ERR_INVALID_ARG
    assert sar.topk_gather_sort(fake, 100, 1, 100, 8, 0, fake) == sar.TOPK_ERR_UNSUPPORTED_TOPK
    assert sar.topk_gather_sort(fake, 100, 1, 100, 0, 512, fake) == sar.TOPK_OK
    assert sar.topk_gather_sort(fake, 100, 1, 100, 8, 512, fake, None, sort=False) == sar.TOPK_OK
    assert sar.topk_gather_sort(fake + 1, 100, 1, 100, 8, 512, fake) == sar.TOPK_ERR_MISALIGNED


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(sar, "_LIB_PATH", str(tmp_path / "libtopk.so"))
    monkeypatch.setattr(sar, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        sar.topk_status_string(0)


def test_binding_structs_match_the_header(tmp_path):
    # the ctypes mirrors of topk_options, topk_device_props and topk_plan must
    # have the header's field offsets and sizes: a C program compiled against
    # include/libtopk.h prints them
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    mirrors = {"topk_options": sar.TopkOptions, "topk_device_props": sar.TopkDeviceProps,
               "topk_plan": sar.TopkPlan}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "libtopk.h"', "int main(void) {"]
    for cname, py in mirrors.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        cname, field, value = line.split()
        got[(cname, field)] = int(value)
    for cname, py in mirrors.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)
