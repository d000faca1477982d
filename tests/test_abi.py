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
