"""CPU checks of the C-ABI boundary: the library builds, loads without a GPU,
exports every call include/pkv.h declares, and the product path contains no
route to the oracle or to any CPU fallback."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
PKG = os.path.join(ROOT, "paged_kv_cache_291_gb300")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_291_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ["pkv_cache_write", "pkv_copy_blocks", "pkv_decode_attention", "pkv_decode_workspace_size",
              "pkv_chunked_prefill_attention", "pkv_prefill_workspace_size", "pkv_get_error", "pkv_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/pkv.h but not exported"


def test_only_pkv_symbols_are_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    extra = [s for s in exported if not s.startswith("pkv_")]
    assert not extra, f"unexpected exported functions: {extra[:10]}"


def test_status_strings_without_gpu(lib):
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(6).startswith(b"PKV_ERR_ALIAS")
    assert lib.pkv_version().count(b".") == 2


def test_binding_status_table_matches_header():
    import paged_kv_cache_291_gb300 as pkv
    text = open(HEADER).read()
    for name, val in re.findall(r"(PKV_(?:OK|ERR_[A-Z]+))\s*=\s*(\d+)", text):
        assert pkv.STATUS_NAMES[int(val)] == name


def test_binding_fails_loudly_without_the_library(tmp_path):
    code = ("import paged_kv_cache_291_gb300 as p; p._LIB_PATH = %r\n"
            "try:\n    p.load()\nexcept RuntimeError as e:\n    print('RAISED', e)\n") % str(tmp_path / "none.so")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "RAISED" in r.stdout and "not built" in r.stdout


def test_product_path_never_touches_the_oracle():
    offenders = []
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                if re.search(r"\boracle\b", text) and re.search(r"import\s+oracle|from\s+oracle|oracle/|liboracle",
                                                                text):
                    offenders.append(f)
    assert not offenders, offenders


def test_sources_use_no_closed_copy_calls():
    pat = re.compile("(cu|cuda)" + "Memcpy" + "(3D)?" + "Batch" + "Async")
    roots = [os.path.join(ROOT, d) for d in ("paged_kv_cache_291_gb300", "include", "oracle", "tests", "pkv_workloads")]
    files = [os.path.join(ROOT, f) for f in ("bench.py", "__graft_entry__.py")]
    for top in roots:
        for dirpath, _, names in os.walk(top):
            if "_build" in dirpath:
                continue
            files += [os.path.join(dirpath, f) for f in names if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp"))]
    for f in files:
        assert not pat.search(open(f, errors="ignore").read()), f


def test_descriptor_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors have the header's field offsets and sizes
    (a C program compiled against include/pkv.h prints them)."""
    import paged_kv_cache_291_gb300 as pkv
    structs = {"pkv_cache_t": pkv.Cache, "pkv_blocks_t": pkv.BlocksState}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "pkv.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append('return 0; }')
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in out if ln}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_e4m3_descriptor_checks_without_gpu(lib):
    """The pool descriptor is checked on the host before anything touches a
    device: an unknown kv_dtype or e4m3 scales that are not finite and
    positive give PKV_ERR_DTYPE (16); a valid e4m3 descriptor with no rows
    is a no-op."""
    import paged_kv_cache_291_gb300 as pkv
    fake = 1 << 20                      # aligned, never dereferenced
    lib.pkv_cache_write.restype = ctypes.c_int

    def write(dtype, ks, vs):
        c = pkv.Cache(fake, fake, 4, 8, 128, 16, dtype, ks, vs)
        return lib.pkv_cache_write(ctypes.byref(c), ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                   ctypes.c_void_p(fake), 0, None)
    assert write(pkv.PKV_KV_E4M3, 0.01, 0.02) == 0
    assert write(pkv.PKV_KV_BF16, 0.0, 0.0) == 0          # scales are ignored for bf16
    assert write(7, 1.0, 1.0) == 16
    for bad in (0.0, -0.5, float("inf"), float("nan"), 1e-45):
        assert write(pkv.PKV_KV_E4M3, bad, 1.0) == 16
        assert write(pkv.PKV_KV_E4M3, 1.0, bad) == 16


def test_copy_argument_checks_without_gpu(lib):
    """pkv_copy checks its arguments before touching a device: 0 bytes is a
    no-op, NULL pointers give PKV_ERR_NULL (1), a size that is not a multiple
    of 16 PKV_ERR_SHAPE (2), unaligned pointers PKV_ERR_ALIGN."""
    import paged_kv_cache_291_gb300 as pkv
    lib.pkv_copy.restype = ctypes.c_int
    lib.pkv_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    a, b = 1 << 20, 2 << 20                 # aligned, never dereferenced
    names = {v: k for k, v in pkv.STATUS_NAMES.items()}
    assert lib.pkv_copy(a, b, 0, None) == 0
    assert lib.pkv_copy(None, b, 16, None) == 1
    assert lib.pkv_copy(a, None, 16, None) == 1
    assert lib.pkv_copy(a, b, 24, None) == 2
    assert lib.pkv_copy(a + 8, b, 16, None) == names["PKV_ERR_ALIGN"]
    assert lib.pkv_copy(a, b + 4, 16, None) == names["PKV_ERR_ALIGN"]
