"""CPU tests of the C-ABI boundary: the library builds, loads without a GPU,
and exports every function include/prnn.h declares (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "prnn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(prnn_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from persistent_rnn_recurrence_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("prnn_create", "prnn_set_weights_dense", "prnn_set_weights_sparse",
              "prnn_forward", "prnn_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header(lib):
    from persistent_rnn_recurrence_gb300 import prnn
    assert sorted(prnn.EXPORTS) == declared_functions()
    for n in prnn.EXPORTS:
        assert callable(getattr(prnn, n))


def test_status_strings_without_gpu(lib):
    from persistent_rnn_recurrence_gb300 import prnn
    assert prnn.prnn_status_string(prnn.PRNN_OK) == "PRNN_OK"
    assert prnn.prnn_status_string(prnn.PRNN_ERR_TIMEOUT) == "PRNN_ERR_TIMEOUT"
    assert prnn.prnn_status_string(99) == "PRNN_ERR_UNKNOWN"


def test_null_arguments_rejected_without_gpu(lib):
    """Argument checks that precede any CUDA call."""
    from persistent_rnn_recurrence_gb300 import prnn
    f = prnn._lib
    assert f.prnn_forward(None, 1, 1, None, None, None, None) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_forward_host(None, 1, 1, None, None, None, None) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_destroy(None) == prnn.PRNN_OK
    assert f.prnn_set_option(None, 0, 1) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_create(None, 8, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert f.prnn_create(ctypes.byref(h), 0, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_create(ctypes.byref(h), 8, 8, 33, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_create(ctypes.byref(h), 8, 8, 1, 7, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert h.value is None


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    """The binding raises ImportError when libprnn.so is absent (no fallback)."""
    import importlib.util
    src = os.path.join(ROOT, "persistent_rnn_recurrence_gb300", "prnn.py")
    dst = tmp_path / "prnn.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("prnn_copy", str(dst))
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_enum_values_match_the_header(lib):
    """Every PRNN_* enumerator of the header has the same value in the binding."""
    from persistent_rnn_recurrence_gb300 import prnn
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    pairs = re.findall(r"\b(PRNN_[A-Z0-9_]+)\s*=\s*(\d+)", text)
    assert len(pairs) >= 25
    for name, value in pairs:
        assert getattr(prnn, name) == int(value), name


def test_struct_layouts_match_the_header(lib, tmp_path):
    """Field offsets and sizes of the info structs as the C compiler lays them
    out from include/prnn.h equal the binding's ctypes mirrors."""
    import shutil
    import subprocess
    from persistent_rnn_recurrence_gb300 import prnn
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "prnn.h"', 'int main(void) {']
    for cname, cls in (("prnn_info_t", prnn.prnn_info_t), ("prnn_stack_info_t", prnn.prnn_stack_info_t)):
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, cls in (("prnn_info_t", prnn.prnn_info_t), ("prnn_stack_info_t", prnn.prnn_stack_info_t)):
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, (cname, f)


def test_stack_and_backward_argument_checks_without_gpu(lib):
    from persistent_rnn_recurrence_gb300 import prnn
    f = prnn._lib
    assert f.prnn_stack_create(None, 2, 8, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    s = ctypes.c_void_p()
    assert f.prnn_stack_create(ctypes.byref(s), 0, 8, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_stack_create(ctypes.byref(s), 9, 8, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_stack_create(ctypes.byref(s), 2, 6, 8, 1, 0, 0) == prnn.PRNN_ERR_INVALID_ARG
    assert s.value is None
    assert f.prnn_stack_destroy(None) == prnn.PRNN_OK
    assert f.prnn_stack_forward(None, 1, 1, None, None, None, None) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_backward(None, 1, 1, None, None, None, None, None, None, None, None, None,
                           None, None) == prnn.PRNN_ERR_INVALID_ARG
    assert f.prnn_set_weights_csr(None, None, 0, None, None, None, None, None) == \
        prnn.PRNN_ERR_INVALID_ARG


def test_cluster_probe_argument_checks_without_gpu(lib):
    """The cluster exchange probe rejects its bad arguments before any CUDA call."""
    from persistent_rnn_recurrence_gb300 import prnn
    f = prnn._lib
    ns, bad = ctypes.c_double(), ctypes.c_longlong()
    out = (ctypes.byref(ns), ctypes.byref(bad))
    for hidden, cs, ncl, steps in ((1792, 3, 1, 10),     # cluster size not 2, 4, 8 or 16
                                   (1790, 4, 1, 10),     # not a multiple of 4 * cluster size
                                   (1800, 16, 1, 10),    # 1800 % 64 != 0
                                   (32, 16, 1, 10),      # fewer than 4 rows per CTA
                                   (20480, 2, 1, 10),    # beyond 16384
                                   (1792, 4, 0, 10),     # no cluster
                                   (1792, 4, 1, 1)):     # fewer than 2 steps
        assert f.prnn_probe_cluster_exchange(hidden, cs, ncl, steps, *out) == \
            prnn.PRNN_ERR_INVALID_ARG, (hidden, cs, ncl, steps)
    assert f.prnn_probe_cluster_exchange(1792, 4, 1, 10, None, ctypes.byref(bad)) == \
        prnn.PRNN_ERR_INVALID_ARG
