"""Thin ctypes binding of libprnn.so (declarations in include/prnn.h).

Every function here marshals arguments and calls the C ABI function of the same
name; every step of the computation runs in the library's CUDA kernels.
PyTorch only supplies device memory and streams.  Importing this module loads
the library and raises ImportError if it has not been built -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libprnn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m persistent_rnn_recurrence_gb300.build`")
_lib = ctypes.CDLL(LIB_PATH)

# ---- enums (mirror include/prnn.h) ------------------------------------------
PRNN_OK, PRNN_ERR_INVALID_ARG, PRNN_ERR_UNSUPPORTED, PRNN_ERR_NOT_READY, \
    PRNN_ERR_CUDA, PRNN_ERR_OOM, PRNN_ERR_TIMEOUT = range(7)
PRNN_F32, PRNN_F16 = 0, 1
PRNN_ALGO_PERSISTENT, PRNN_ALGO_PER_STEP = 0, 1
(PRNN_OPT_WAIT_TIMEOUT_US, PRNN_OPT_SYNC_MODE, PRNN_OPT_DEBUG_DROP_CTA,
 PRNN_OPT_DEBUG_DROP_STEP, PRNN_OPT_TIMING, PRNN_OPT_PROJECTION, PRNN_OPT_CTA_GROUPS,
 PRNN_OPT_WIDE_LOADS, PRNN_OPT_BANK_AWARE, PRNN_OPT_POLL_DELAY_NS,
 PRNN_OPT_POLL_BACKOFF_NS, PRNN_OPT_RECURRENT_TC, PRNN_OPT_STAGED_ORDER,
 PRNN_OPT_SPARSE_REG_WEIGHTS, PRNN_OPT_SPARSE_STAGING_DEPTH, PRNN_OPT_DENSE_WIDE,
 PRNN_OPT_DENSE_KSPLIT, PRNN_OPT_SPARSE_KSPLIT) = range(18)

PRNN_STACK_WAVEFRONT, PRNN_STACK_LAYERWISE = 0, 1

EXPORTS = ["prnn_create", "prnn_set_weights_dense", "prnn_set_weights_sparse",
           "prnn_forward", "prnn_forward_host", "prnn_destroy", "prnn_get_status", "prnn_status_string",
           "prnn_set_option", "prnn_get_info", "prnn_get_timing", "prnn_probe_sync_floor",
           "prnn_probe_cluster_exchange",
           "prnn_set_trace_buffer",
           "prnn_pack_sparse_host", "prnn_pack_sparse_host_placed", "prnn_pack_dense_ksplit_host",
           "prnn_forward_dense_noalloc",
           "prnn_set_weights_csr",
           "prnn_stack_create", "prnn_stack_set_layer", "prnn_stack_forward",
           "prnn_stack_get_status", "prnn_stack_set_option", "prnn_stack_get_timing",
           "prnn_stack_get_info", "prnn_stack_destroy", "prnn_backward"]


class prnn_info_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "hidden", "input", "max_batch", "wdtype", "algo", "sparse", "weights_set", "k",
        "k_padded", "sm_count", "n_cta", "rows_per_cta", "threads_per_cta",
        "threads_per_row", "projection_tensor_cores", "sparse_bank_cap", "cta_groups")] + [
        ("smem_bytes", ctypes.c_size_t), ("onchip_weight_bytes", ctypes.c_size_t),
        ("nnz", ctypes.c_size_t), ("recurrent_tensor_cores", ctypes.c_int),
        ("sparse_staged_order", ctypes.c_int), ("sparse_reg_weights", ctypes.c_int),
        ("dense_wide_batch", ctypes.c_int), ("dense_ksplit", ctypes.c_int)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class prnn_stack_info_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "layers", "hidden", "input", "max_batch", "wdtype", "algo", "layers_set",
        "n_cta_per_layer", "rows_per_cta", "threads_per_cta", "cta_groups", "batch_per_pass",
        "chunks_per_thread")] + [
        ("smem_bytes", ctypes.c_longlong), ("onchip_weight_bytes", ctypes.c_longlong)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_P = ctypes.c_void_p
_I = ctypes.c_int
_sig = {
    "prnn_create": ([ctypes.POINTER(_P), _I, _I, _I, _I, _I], _I),
    "prnn_set_weights_dense": ([_P, _P, _P, _P, _P], _I),
    "prnn_set_weights_sparse": ([_P, _P, _I, _P, _P, _P, _P], _I),
    "prnn_forward": ([_P, _I, _I, _P, _P, _P, _P], _I),
    "prnn_forward_host": ([_P, _I, _I, _P, _P, _P, _P], _I),
    "prnn_destroy": ([_P], _I),
    "prnn_get_status": ([_P, _P], _I),
    "prnn_status_string": ([_I], ctypes.c_char_p),
    "prnn_set_option": ([_P, _I, ctypes.c_longlong], _I),
    "prnn_get_info": ([_P, ctypes.POINTER(prnn_info_t)], _I),
    "prnn_get_timing": ([_P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)], _I),
    "prnn_probe_sync_floor": ([_P, _I, _I, _P, _P], _I),
    "prnn_probe_cluster_exchange": ([_I, _I, _I, _I, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_longlong)], _I),
    "prnn_set_trace_buffer": ([_P, _P, ctypes.c_size_t], _I),
    "prnn_pack_sparse_host": ([_I, _I, _I, _I, _I, _P, _P, _P, ctypes.c_size_t,
                               ctypes.POINTER(_I), ctypes.POINTER(_I)], _I),
    "prnn_pack_sparse_host_placed": ([_I, _I, _I, _I, _I, _P, _P, _P, ctypes.c_size_t, _P,
                                      ctypes.c_size_t, ctypes.POINTER(_I), ctypes.POINTER(_I),
                                      ctypes.POINTER(_I)], _I),
    "prnn_pack_dense_ksplit_host": ([_I, _I, _P, _I, _P, ctypes.c_size_t,
                                     ctypes.POINTER(ctypes.c_size_t)], _I),
    "prnn_forward_dense_noalloc": ([_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P], _I),
    "prnn_set_weights_csr": ([_P, _P, _I, _P, _P, _P, _P, _P], _I),
    "prnn_stack_create": ([ctypes.POINTER(_P), _I, _I, _I, _I, _I, _I], _I),
    "prnn_stack_set_layer": ([_P, _I, _P, _P, _P, _P], _I),
    "prnn_stack_forward": ([_P, _I, _I, _P, _P, _P, _P], _I),
    "prnn_stack_get_status": ([_P, _P], _I),
    "prnn_stack_set_option": ([_P, _I, ctypes.c_longlong], _I),
    "prnn_stack_get_timing": ([_P, ctypes.POINTER(ctypes.c_float)], _I),
    "prnn_stack_get_info": ([_P, ctypes.POINTER(prnn_stack_info_t)], _I),
    "prnn_stack_destroy": ([_P], _I),
    "prnn_backward": ([_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
}
for _name, (_args, _res) in _sig.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class PrnnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {prnn_status_string(status)}")


def prnn_status_string(status: int) -> str:
    return _lib.prnn_status_string(int(status)).decode()


def _check(status: int, where: str) -> int:
    if status != PRNN_OK:
        raise PrnnError(status, where)
    return status


def _ptr(t) -> Optional[int]:
    """Device/host address of a tensor (or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- the C ABI, one Python function per C function ---------------------------
def prnn_create(hidden: int, input: int, max_batch: int, wdtype: int, algo: int) -> int:
    h = _P()
    _check(_lib.prnn_create(ctypes.byref(h), hidden, input, max_batch, wdtype, algo),
           "prnn_create")
    return h.value


def prnn_set_weights_dense(h: int, Wx, Wh, bias, stream=None) -> None:
    _check(_lib.prnn_set_weights_dense(h, _ptr(Wx), _ptr(Wh), _ptr(bias), _stream(stream)),
           "prnn_set_weights_dense")


def prnn_set_weights_sparse(h: int, Wx, k: int, vals, cols, bias, stream=None) -> None:
    _check(_lib.prnn_set_weights_sparse(h, _ptr(Wx), int(k), _ptr(vals), _ptr(cols),
                                        _ptr(bias), _stream(stream)),
           "prnn_set_weights_sparse")


def prnn_set_weights_csr(h: int, Wx, nnz: int, row_ptr, cols, vals, bias, stream=None) -> None:
    _check(_lib.prnn_set_weights_csr(h, _ptr(Wx), int(nnz), _ptr(row_ptr), _ptr(cols),
                                     _ptr(vals), _ptr(bias), _stream(stream)),
           "prnn_set_weights_csr")


def prnn_forward(h: int, T: int, B: int, x, h0, y, stream=None) -> None:
    _check(_lib.prnn_forward(h, T, B, _ptr(x), _ptr(h0), _ptr(y), _stream(stream)),
           "prnn_forward")


def prnn_forward_host(h: int, T: int, B: int, x, h0, y, stream=None) -> None:
    """x, h0 (or None) and y are page-locked host buffers (e.g. pinned CPU
    tensors)."""
    _check(_lib.prnn_forward_host(h, T, B, _ptr(x), _ptr(h0), _ptr(y), _stream(stream)),
           "prnn_forward_host")


def prnn_destroy(h: int) -> None:
    _check(_lib.prnn_destroy(h), "prnn_destroy")


def prnn_get_status(h: int, stream=None) -> int:
    """Returns the status code (PRNN_OK or PRNN_ERR_TIMEOUT); does not raise
    for a timeout, so callers can test for it."""
    return _lib.prnn_get_status(h, _stream(stream))


def prnn_set_option(h: int, opt: int, value: int) -> None:
    _check(_lib.prnn_set_option(h, opt, int(value)), "prnn_set_option")


def prnn_get_info(h: int) -> dict:
    info = prnn_info_t()
    _check(_lib.prnn_get_info(h, ctypes.byref(info)), "prnn_get_info")
    return info.as_dict()


def prnn_get_timing(h: int):
    a, b = ctypes.c_float(), ctypes.c_float()
    _check(_lib.prnn_get_timing(h, ctypes.byref(a), ctypes.byref(b)), "prnn_get_timing")
    return a.value, b.value


def prnn_pack_sparse_host_placed(hidden, k, n_cta, rows_per_cta, threads_per_row, vals, cols):
    """Host-only packing with the per-CTA staging order of h: returns
    (packed[n_cta, R, ept/4, tpr, 4] uint32, place[n_cta, hidden/4] uint32 or
    None when columns stay in order, ept, bank_cap)."""
    import numpy as np
    vals = np.ascontiguousarray(vals).view(np.uint16)
    cols = np.ascontiguousarray(cols, dtype=np.uint16)
    ept, cap, placed = _I(), _I(), _I()
    st = _lib.prnn_pack_sparse_host_placed(hidden, k, n_cta, rows_per_cta, threads_per_row,
                                           vals.ctypes.data, cols.ctypes.data, None, 0, None, 0,
                                           ctypes.byref(ept), ctypes.byref(cap),
                                           ctypes.byref(placed))
    if st != PRNN_ERR_INVALID_ARG or ept.value <= 0:
        _check(st if st != PRNN_OK else PRNN_ERR_INVALID_ARG, "prnn_pack_sparse_host_placed")
    out = np.zeros((n_cta, rows_per_cta, ept.value // 4, threads_per_row, 4), dtype=np.uint32)
    place = np.zeros((n_cta, hidden // 4), dtype=np.uint32) if placed.value else None
    _check(_lib.prnn_pack_sparse_host_placed(
        hidden, k, n_cta, rows_per_cta, threads_per_row, vals.ctypes.data, cols.ctypes.data,
        out.ctypes.data, out.size, None if place is None else place.ctypes.data,
        0 if place is None else place.size, ctypes.byref(ept), ctypes.byref(cap),
        ctypes.byref(placed)), "prnn_pack_sparse_host_placed")
    return out, place, ept.value, cap.value


def prnn_probe_sync_floor(h: int, T: int, B: int, y, stream=None) -> None:
    _check(_lib.prnn_probe_sync_floor(h, T, B, _ptr(y), _stream(stream)),
           "prnn_probe_sync_floor")


def prnn_probe_cluster_exchange(hidden: int, cluster_size: int, clusters: int,
                                steps: int) -> tuple:
    """(ns per step, wrong words received) of the cluster exchange probe."""
    ns = ctypes.c_double(0.0)
    bad = ctypes.c_longlong(0)
    _check(_lib.prnn_probe_cluster_exchange(hidden, cluster_size, clusters, steps,
                                            ctypes.byref(ns), ctypes.byref(bad)),
           "prnn_probe_cluster_exchange")
    return ns.value, bad.value


def prnn_set_trace_buffer(h: int, buf, nbytes: int) -> None:
    """Set (or, with buf None, clear) the device buffer of the sparse
    kernel's phase trace: [T][n_cta][12] uint32 records per forward."""
    _check(_lib.prnn_set_trace_buffer(h, _ptr(buf), int(nbytes)), "prnn_set_trace_buffer")


def prnn_pack_dense_ksplit_host(hidden, cluster_size, wh16, transpose=False):
    """Host-only image of the K-split kernel's weights (numpy fp16 [H, H] in,
    numpy uint16 [H/128, cluster_size, nat, 128, 64] out)."""
    import numpy as np
    w = np.ascontiguousarray(wh16).view(np.uint16)
    if w.shape != (hidden, hidden):
        raise ValueError("wh16 must be [hidden, hidden]")
    need = ctypes.c_size_t()
    st = _lib.prnn_pack_dense_ksplit_host(hidden, cluster_size, w.ctypes.data, int(transpose),
                                          None, 0, ctypes.byref(need))
    if st != PRNN_ERR_INVALID_ARG or need.value == 0:
        _check(st if st != PRNN_OK else PRNN_ERR_INVALID_ARG, "prnn_pack_dense_ksplit_host")
    nat = need.value // ((hidden // 128) * cluster_size * 8192)
    out = np.zeros((hidden // 128, cluster_size, nat, 128, 64), dtype=np.uint16)
    _check(_lib.prnn_pack_dense_ksplit_host(hidden, cluster_size, w.ctypes.data, int(transpose),
                                            out.ctypes.data, out.size, ctypes.byref(need)),
           "prnn_pack_dense_ksplit_host")
    return out


def prnn_pack_sparse_host(hidden, k, n_cta, rows_per_cta, threads_per_row, vals, cols):
    """Host-only packing (numpy in, numpy out): returns (packed[n_cta, R, ept/4,
    tpr, 4] uint32, ept, bank_cap)."""
    import numpy as np
    vals = np.ascontiguousarray(vals).view(np.uint16)
    cols = np.ascontiguousarray(cols, dtype=np.uint16)
    ept, cap = _I(), _I()
    st = _lib.prnn_pack_sparse_host(hidden, k, n_cta, rows_per_cta, threads_per_row,
                                    vals.ctypes.data, cols.ctypes.data, None, 0,
                                    ctypes.byref(ept), ctypes.byref(cap))
    if st != PRNN_ERR_INVALID_ARG or ept.value <= 0:
        _check(st if st != PRNN_OK else PRNN_ERR_INVALID_ARG, "prnn_pack_sparse_host")
    out = np.zeros((n_cta, rows_per_cta, ept.value // 4, threads_per_row, 4), dtype=np.uint32)
    _check(_lib.prnn_pack_sparse_host(hidden, k, n_cta, rows_per_cta, threads_per_row,
                                      vals.ctypes.data, cols.ctypes.data, out.ctypes.data,
                                      out.size, ctypes.byref(ept), ctypes.byref(cap)),
           "prnn_pack_sparse_host")
    return out, ept.value, cap.value


def prnn_forward_dense_noalloc(T, B, H, I, wdtype, x, Wx, Wh, bias, h0, y, stream=None) -> None:
    """Dense forward from the caller's own device buffers, allocating nothing
    (see include/prnn.h for the scratch limits and the sharing rules)."""
    _check(_lib.prnn_forward_dense_noalloc(T, B, H, I, wdtype, _ptr(x), _ptr(Wx), _ptr(Wh),
                                           _ptr(bias), _ptr(h0), _ptr(y), _stream(stream)),
           "prnn_forward_dense_noalloc")


def prnn_backward(h: int, T: int, B: int, x, h0, y, dy, delta=None, dx=None, dh0=None, dWx=None,
                  dWh=None, db=None, stream=None) -> None:
    _check(_lib.prnn_backward(h, T, B, _ptr(x), _ptr(h0), _ptr(y), _ptr(dy), _ptr(delta), _ptr(dx),
                              _ptr(dh0), _ptr(dWx), _ptr(dWh), _ptr(db), _stream(stream)),
           "prnn_backward")


def prnn_stack_create(layers: int, hidden: int, input: int, max_batch: int, wdtype: int,
                      algo: int) -> int:
    out = _P()
    _check(_lib.prnn_stack_create(ctypes.byref(out), layers, hidden, input, max_batch, wdtype,
                                  algo), "prnn_stack_create")
    return out.value


def prnn_stack_set_layer(s: int, layer: int, Wx, Wh, bias, stream=None) -> None:
    _check(_lib.prnn_stack_set_layer(s, layer, _ptr(Wx), _ptr(Wh), _ptr(bias), _stream(stream)),
           "prnn_stack_set_layer")


def prnn_stack_forward(s: int, T: int, B: int, x, h0, y, stream=None) -> None:
    _check(_lib.prnn_stack_forward(s, T, B, _ptr(x), _ptr(h0), _ptr(y), _stream(stream)),
           "prnn_stack_forward")


def prnn_stack_get_status(s: int, stream=None) -> int:
    return _lib.prnn_stack_get_status(s, _stream(stream))


def prnn_stack_set_option(s: int, opt: int, value: int) -> None:
    _check(_lib.prnn_stack_set_option(s, opt, int(value)), "prnn_stack_set_option")


def prnn_stack_get_timing(s: int) -> float:
    ms = ctypes.c_float()
    _check(_lib.prnn_stack_get_timing(s, ctypes.byref(ms)), "prnn_stack_get_timing")
    return ms.value


def prnn_stack_get_info(s: int) -> dict:
    info = prnn_stack_info_t()
    _check(_lib.prnn_stack_get_info(s, ctypes.byref(info)), "prnn_stack_get_info")
    return info.as_dict()


def prnn_stack_destroy(s: int) -> None:
    _check(_lib.prnn_stack_destroy(s), "prnn_stack_destroy")


# ---- convenience wrapper used by the tests and the benchmark ------------------
class Layer:
    """One RNN layer handle.  ``Layer.from_problem(p)`` uploads a
    ``synth.Problem``'s weights (as device tensors) and returns the layer."""

    def __init__(self, hidden, input, max_batch, wdtype="f16", algo="persistent"):
        self.hidden, self.input, self.max_batch = hidden, input, max_batch
        wd = {"f32": PRNN_F32, "f16": PRNN_F16}[wdtype]
        al = {"persistent": PRNN_ALGO_PERSISTENT, "per_step": PRNN_ALGO_PER_STEP}[algo]
        self.h = prnn_create(hidden, input, max_batch, wd, al)

    @classmethod
    def from_problem(cls, p, algo="persistent", max_batch=None, device="cuda"):
        import torch
        lay = cls(p.H, p.I, max_batch or max(1, p.B), p.wdtype, algo)
        try:
            lay.set_problem_weights(p, device)
        except Exception:
            lay.close()
            raise
        return lay

    def set_problem_weights(self, p, device="cuda"):
        import numpy as np
        import torch
        wt = torch.float16 if p.wdtype == "f16" else torch.float32
        Wx = torch.from_numpy(np.ascontiguousarray(p.Wx)).to(device=device, dtype=wt)
        b = torch.from_numpy(np.ascontiguousarray(p.b)).to(device)
        if getattr(p, "row_ptr", None) is not None:
            rp = torch.from_numpy(np.ascontiguousarray(p.row_ptr, dtype=np.int32)).to(device)
            vals = torch.from_numpy(np.ascontiguousarray(p.vals).view(np.int16)).to(device)
            cols = torch.from_numpy(np.ascontiguousarray(p.cols).view(np.int16)).to(device)
            prnn_set_weights_csr(self.h, Wx, int(p.vals.size), rp, cols, vals, b)
            self.n_values = int(p.vals.size)
        elif p.sparse:
            vals = torch.from_numpy(np.ascontiguousarray(p.vals).view(np.int16)).to(device)
            cols = torch.from_numpy(np.ascontiguousarray(p.cols).view(np.int16)).to(device)
            prnn_set_weights_sparse(self.h, Wx, p.k, vals, cols, b)
        else:
            Wh = torch.from_numpy(np.ascontiguousarray(p.Wh)).to(device=device, dtype=wt)
            prnn_set_weights_dense(self.h, Wx, Wh, b)
        torch.cuda.synchronize()

    def forward(self, x, h0=None, y=None, stream=None):
        """x: [T,B,I] fp32 CUDA tensor; returns y [T,B,H] fp32."""
        import torch
        T, B, _ = x.shape
        if y is None:
            y = torch.empty((T, B, self.hidden), dtype=torch.float32, device=x.device)
        prnn_forward(self.h, T, B, x, h0, y, stream)
        return y

    def backward(self, x, y, dy, h0=None, stream=None) -> dict:
        """Gradients of the loss with dL/dy = dy for the forward (x, h0) -> y:
        dict of fp32 CUDA tensors delta, dx, dh0, dWx, dWh, db."""
        import torch
        T, B, _ = x.shape
        dev = x.device
        info = self.info()
        if info["sparse"]:
            nv = self.n_values if getattr(self, "n_values", None) else info["hidden"] * info["k"]
            dwh = torch.empty(nv, device=dev)
        else:
            dwh = torch.empty(self.hidden, self.hidden, device=dev)
        g = {"delta": torch.empty_like(y),
             "dx": torch.empty_like(x), "dh0": torch.empty(B, self.hidden, device=dev),
             "dWx": torch.empty(self.hidden, self.input, device=dev), "dWh": dwh,
             "db": torch.empty(self.hidden, device=dev)}
        prnn_backward(self.h, T, B, x, h0, y, dy, g["delta"], g["dx"], g["dh0"], g["dWx"], g["dWh"],
                      g["db"], stream)
        return g

    def status(self, stream=None) -> int:
        return prnn_get_status(self.h, stream)

    def info(self) -> dict:
        return prnn_get_info(self.h)

    def set_option(self, opt, value):
        prnn_set_option(self.h, opt, value)

    def close(self):
        if getattr(self, "h", None):
            prnn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Stack:
    """A stack of dense layers (``prnn_stack_*``).  ``Stack.from_problem(p)``
    uploads a ``synth.StackProblem``'s weights and returns the stack."""

    def __init__(self, layers, hidden, input, max_batch, wdtype="f16", algo="wavefront"):
        self.layers, self.hidden, self.input = layers, hidden, input
        wd = {"f32": PRNN_F32, "f16": PRNN_F16}[wdtype]
        al = {"wavefront": PRNN_STACK_WAVEFRONT, "layerwise": PRNN_STACK_LAYERWISE}[algo]
        self.h = prnn_stack_create(layers, hidden, input, max_batch, wd, al)

    @classmethod
    def from_problem(cls, p, algo="wavefront", max_batch=None, device="cuda"):
        st = cls(p.L, p.H, p.I, max_batch or max(1, p.B), p.wdtype, algo)
        try:
            st.set_problem_weights(p, device)
        except Exception:
            st.close()
            raise
        return st

    def set_problem_weights(self, p, device="cuda"):
        import numpy as np
        import torch
        wt = torch.float16 if p.wdtype == "f16" else torch.float32
        for l, (Wx, Wh, b) in enumerate(p.layers):
            prnn_stack_set_layer(
                self.h, l, torch.from_numpy(np.ascontiguousarray(Wx)).to(device=device, dtype=wt),
                torch.from_numpy(np.ascontiguousarray(Wh)).to(device=device, dtype=wt),
                torch.from_numpy(np.ascontiguousarray(b)).to(device))
        torch.cuda.synchronize()

    def forward(self, x, h0=None, y=None, stream=None):
        """x: [T,B,I] fp32 CUDA tensor; returns y [L,T,B,H] (every layer's output)."""
        import torch
        T, B, _ = x.shape
        if y is None:
            y = torch.empty((self.layers, T, B, self.hidden), dtype=torch.float32, device=x.device)
        prnn_stack_forward(self.h, T, B, x, h0, y, stream)
        return y

    def status(self, stream=None) -> int:
        return prnn_stack_get_status(self.h, stream)

    def info(self) -> dict:
        return prnn_stack_get_info(self.h)

    def set_option(self, opt, value):
        prnn_stack_set_option(self.h, opt, value)

    def close(self):
        if getattr(self, "h", None):
            prnn_stack_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
