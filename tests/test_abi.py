"""The C-ABI library builds, loads and exports every symbol include/nvfp4_mla.h declares;
argument checks that need no device return their status codes. No kernel runs here."""
import ctypes
import os
import re

import pytest

import nvfp4_kv_cache_sparse_gb300 as lib
from nvfp4_kv_cache_sparse_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4_mla.h")


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"NVFP4_MLA_API\s+[\w\s\*]+?\b(nvfp4_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def cdll():
    build.build()
    return lib.load()


def test_header_declares_the_expected_calls():
    syms = declared_symbols()
    assert set(syms) == set(lib.EXPORTED), syms


def test_header_compiles_as_strict_c99(tmp_path):
    # the boundary is a C ABI: the header must stand alone in a C translation unit
    src = tmp_path / "use_header.c"
    src.write_text('#include "nvfp4_mla.h"\n'
                   "int main(void) {\n"
                   "    size_t n = 0;\n"
                   "    return nvfp4_sparse_mla_decode_workspace_size(1, 1, 64, 64, 352, 1, &n);\n"
                   "}\n")
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_a_c_program_links_and_calls_the_host_side_entry_points(tmp_path, cdll):
    # a C caller, linked against the shared library, gets the documented host-side answers
    # (no call here needs a GPU)
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "nvfp4_mla.h"
int main(void) {
    size_t n = 1;
    if (nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 352, 1, &n) != NVFP4_MLA_OK || n != 0) return 1;
    if (nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 656, 2, &n) != NVFP4_MLA_OK ||
        n != (size_t)2 * 2 * 64 * 512 * 2 + 1024) return 2;
    if (nvfp4_sparse_mla_decode_workspace_size(1, 1, 64, 64, 400, 1, &n) != NVFP4_MLA_ERR_UNSUPPORTED) return 3;
    if (nvfp4_mla_quantize_append(NULL, 512, NULL, 64, NULL, 0, NULL, 0, 352, NULL, NULL) != NVFP4_MLA_OK) return 4;
    if (nvfp4_mla_status_string(NVFP4_MLA_OK) == NULL || nvfp4_mla_version() <= 0) return 5;
    printf("ok %s\n", nvfp4_mla_status_string(NVFP4_MLA_ERR_WORKSPACE));
    return 0;
}
""")
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(lib.library_path())
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        "-L", libdir, "-lnvfp4mla", "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.startswith("ok "), (run.returncode, run.stdout, run.stderr)


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define NVFP4_MLA_SCALES_BLOCK_ORDER (0x[0-9a-fA-F]+)", text)
    assert m and int(m.group(1), 16) == lib.SCALES_BLOCK_ORDER
    m = re.search(r"#define NVFP4_MLA_NO_ALLOC_SCRATCH_BYTES \(\(\(size_t\)(\d+)\) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == lib.NO_ALLOC_SCRATCH_BYTES
    for name, value in (("SLOT_OUT_OF_RANGE", lib.DEV_SLOT_OUT_OF_RANGE), ("INDEX_OUT_OF_RANGE", lib.DEV_INDEX_OUT_OF_RANGE),
                        ("TIMEOUT", lib.DEV_TIMEOUT), ("FP8_RANGE", lib.DEV_FP8_RANGE)):
        m = re.search(r"#define NVFP4_MLA_DEV_%s (0x[0-9a-fA-F]+)u" % name, text)
        assert m and int(m.group(1), 16) == value, name


def test_library_exports_every_declared_symbol(cdll):
    for name in declared_symbols():
        assert hasattr(cdll, name), name
    nm = os.popen(f"nm -D --defined-only {build.LIB}").read()
    exported = set(re.findall(r"\bT (nvfp4_\w+)", nm))
    assert exported == set(declared_symbols())


def test_status_strings_and_version(cdll):
    for code in range(5):
        assert isinstance(lib.status_string(code), str) and lib.status_string(code)
    assert lib.status_string(99) == "unknown status"
    assert cdll.nvfp4_mla_version() == 100


def test_host_side_checks_return_codes_without_a_device(cdll):
    # unsupported record width / head count are rejected before any CUDA call
    n = ctypes.c_size_t(123)
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(1, 1, 64, 64, 400, 1, ctypes.byref(n)) == lib.ERR_UNSUPPORTED
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(1, 1, 96, 64, 352, 1, ctypes.byref(n)) == lib.ERR_UNSUPPORTED
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(1, 1, 64, 0, 352, 1, ctypes.byref(n)) == lib.ERR_INVALID_ARG
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(1, 1, 64, 64, 352, 65, ctypes.byref(n)) == lib.ERR_INVALID_ARG
    # an explicit split count needs no device: workspace = partial outputs + lse (256-B padded)
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 352, 1, ctypes.byref(n)) == lib.OK and n.value == 0
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 352, 2, ctypes.byref(n)) == lib.OK
    assert n.value == 2 * 2 * 64 * 512 * 2 + 1024
    # quantize_append: zero tokens is a no-op; bad record width / null pointers are errors
    assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 0, None, 0, 352, None, None) == lib.OK
    assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 4, None, 8, 352, None, None) == lib.ERR_INVALID_ARG
    assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 4, None, 8, 353, None, None) == lib.ERR_UNSUPPORTED
    # the 656-byte fp8 record
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 656, 2, ctypes.byref(n)) == lib.OK
    assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 4, None, 8, 656, None, None) == lib.ERR_INVALID_ARG
    # the block-order scale layout exists for the 352-byte record only
    blk = lib.SCALES_BLOCK_ORDER
    assert cdll.nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, 352 | blk, 2, ctypes.byref(n)) == lib.OK
    assert n.value == 2 * 2 * 64 * 512 * 2 + 1024
    for bad in (432 | blk, 656 | blk, 352 | 0x20000, blk):
        assert cdll.nvfp4_sparse_mla_decode_workspace_size(2, 1, 64, 64, bad, 2, ctypes.byref(n)) == lib.ERR_UNSUPPORTED
        assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 4, None, 8, bad, None, None) == lib.ERR_UNSUPPORTED
    assert cdll.nvfp4_mla_quantize_append(None, 512, None, 64, None, 4, None, 8, 352 | blk, None, None) == lib.ERR_INVALID_ARG
    # the no-allocation decode checks its arguments first, like the workspace entry point (its
    # scratch limit, ERR_WORKSPACE, is checked on a GPU in test_zz_no_alloc.py)
    big = 64 * 64 * 128 * 512 * 2                 # 64 rows x 64 splits x 128 heads of f16 partials
    assert big > lib.NO_ALLOC_SCRATCH_BYTES
    assert cdll.nvfp4_sparse_mla_decode_no_alloc(None, None, 8, 352, None, 64, 1, 128, 4096, 1.0, None, None, None,
                                                 64, None, None) == lib.ERR_INVALID_ARG
    assert cdll.nvfp4_sparse_mla_decode_no_alloc(None, None, 8, 400, None, 1, 1, 128, 64, 1.0, None, None, None,
                                                 1, None, None) == lib.ERR_UNSUPPORTED
    # decode: null pointers
    assert cdll.nvfp4_sparse_mla_decode(None, None, 8, 352, None, 1, 1, 64, 64, 1.0, None, None, None, 1, None, 0,
                                        None, None) == lib.ERR_INVALID_ARG
