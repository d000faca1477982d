"""ctypes front end of the fp64 CPU oracle (``prnn_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the CUDA library and its
Python binding never do, and share no code with it.

Every input is widened to float64 exactly (fp16 and fp32 values are exactly
representable in fp64), so the oracle sees the same numbers the GPU path is
given.  What the C side computes, and the passages it follows, is stated in the
header of ``prnn_oracle.c``.

Parity pins: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (hand-computed steps, closed forms, exact
rational brute force, the linear regime, homogeneity, chaining, sparse and
compressed-row versus densified equality, stacking identities, and for the
backward pass exact-rational central differences of the loss and the linear
regime of the reverse recurrence) -- none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "prnn_oracle.c")
LIB = os.path.join(_HERE, "_build", "liboracle.so")

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.POINTER(ctypes.c_long)
_l = ctypes.c_long


def compile_oracle(source: str = SOURCE, out: str = LIB) -> str:
    """Compile the C oracle with gcc into a shared library and return its path.
    Floating-point contraction is off so that x86 and Arm hosts give the same
    bits."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-pthread",
           "-shared", "-fPIC", "-o", out, source]
    subprocess.run(cmd, check=True)
    return out


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: Optional[np.ndarray], t=_D):
    return None if a is None else a.ctypes.data_as(t)


class Oracle:
    """The fp64 reference.  ``Oracle(path)`` loads a given build of it (the
    mutation tests load deliberately broken copies)."""

    def __init__(self, lib_path: str = LIB):
        if lib_path == LIB:
            if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SOURCE):
                compile_oracle()
        elif not os.path.exists(lib_path):
            raise FileNotFoundError(lib_path)
        self.lib = ctypes.CDLL(lib_path)
        L = self.lib
        L.oracle_rnn_forward_dense.argtypes = [_l, _l, _l, _l, _D, _D, _D, _D, _D, _D]
        L.oracle_rnn_forward_dense.restype = ctypes.c_int
        L.oracle_rnn_forward_sparse.argtypes = [_l, _l, _l, _l, _l, _D, _D, _D, _L, _D,
                                                _D, _D]
        L.oracle_rnn_forward_sparse.restype = ctypes.c_int
        L.oracle_rnn_forward_threads.argtypes = [_l, _l, _l, _l, _l, _D, _D, _D, _D, _L, _D,
                                                 _D, _D, _l]
        L.oracle_rnn_forward_threads.restype = ctypes.c_int
        L.oracle_rnn_input_projection.argtypes = [_l, _l, _l, _l, _D, _D, _D, _D]
        L.oracle_rnn_input_projection.restype = ctypes.c_int
        L.oracle_rnn_cell_dense.argtypes = [_l, _l, _l, _D, _D, _D, _D, _D]
        L.oracle_rnn_cell_dense.restype = ctypes.c_double
        L.oracle_rnn_cell_sparse.argtypes = [_l, _l, _l, _l, _D, _D, _D, _L, _D, _D]
        L.oracle_rnn_cell_sparse.restype = ctypes.c_double
        L.oracle_rnn_forward_csr.argtypes = [_l, _l, _l, _l, _D, _D, _L, _D, _L, _D, _D, _D]
        L.oracle_rnn_forward_csr.restype = ctypes.c_int
        L.oracle_rnn_cell_csr.argtypes = [_l, _l, _l, _D, _D, _L, _D, _L, _D, _D]
        L.oracle_rnn_cell_csr.restype = ctypes.c_double
        L.oracle_rnn_backward_dense.argtypes = [_l, _l, _l, _l, _D, _D, _D, _D, _D, _D, _D, _D,
                                                _D, _D, _D, _D]
        L.oracle_rnn_backward_dense.restype = ctypes.c_int
        L.oracle_rnn_delta_cell_dense.argtypes = [_l, _l, _D, _D, _D, _D]
        L.oracle_rnn_delta_cell_dense.restype = ctypes.c_double

    # -- whole sequences -------------------------------------------------
    def forward_dense(self, x, Wx, Wh, b, h0=None) -> np.ndarray:
        """y[T,B,H] for dense Wh[H,H]; x[T,B,I], Wx[H,I], b[H], h0[B,H]|None."""
        x, Wx, Wh, b = _f64(x), _f64(Wx), _f64(Wh), _f64(b)
        T, B, I = x.shape
        H = Wh.shape[0]
        assert Wx.shape == (H, I) and Wh.shape == (H, H) and b.shape == (H,)
        h0 = None if h0 is None else _f64(h0)
        assert h0 is None or h0.shape == (B, H)
        y = np.zeros((T, B, H), dtype=np.float64)
        rc = self.lib.oracle_rnn_forward_dense(T, B, H, I, _ptr(x), _ptr(Wx), _ptr(Wh),
                                               _ptr(b), _ptr(h0), _ptr(y))
        if rc != 0:
            raise ValueError("oracle_rnn_forward_dense rejected its arguments")
        return y

    def forward_sparse(self, x, Wx, vals, cols, b, h0=None) -> np.ndarray:
        """y[T,B,H] for row-balanced Wh given as vals[H,k], cols[H,k]."""
        x, Wx, vals, b = _f64(x), _f64(Wx), _f64(vals), _f64(b)
        cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        T, B, I = x.shape
        H, k = vals.shape
        assert cols.shape == (H, k) and Wx.shape == (H, I) and b.shape == (H,)
        h0 = None if h0 is None else _f64(h0)
        assert h0 is None or h0.shape == (B, H)
        y = np.zeros((T, B, H), dtype=np.float64)
        rc = self.lib.oracle_rnn_forward_sparse(T, B, H, I, k, _ptr(x), _ptr(Wx),
                                                _ptr(vals), _ptr(cols, _L), _ptr(b),
                                                _ptr(h0), _ptr(y))
        if rc != 0:
            raise ValueError("oracle_rnn_forward_sparse rejected its arguments")
        return y

    def forward_threads(self, x, Wx, b, h0=None, *, Wh=None, vals=None, cols=None,
                        threads: int = 1) -> np.ndarray:
        """The dense (``Wh``) or row-balanced sparse (``vals``, ``cols``) forward
        with each step's outputs split over ``threads`` host threads; the same
        cell arithmetic as the one-thread drivers, so the same bits."""
        x, Wx, b = _f64(x), _f64(Wx), _f64(b)
        T, B, I = x.shape
        H = Wx.shape[0]
        assert b.shape == (H,) and (Wh is None) != (vals is None)
        k = 0
        if Wh is not None:
            Wh = _f64(Wh)
            assert Wh.shape == (H, H)
        else:
            vals = _f64(vals)
            cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
            k = vals.shape[1]
            assert vals.shape == (H, k) and cols.shape == (H, k)
        h0 = None if h0 is None else _f64(h0)
        assert h0 is None or h0.shape == (B, H)
        y = np.zeros((T, B, H), dtype=np.float64)
        rc = self.lib.oracle_rnn_forward_threads(T, B, H, I, k, _ptr(x), _ptr(Wx), _ptr(Wh),
                                                 _ptr(vals), _ptr(cols, _L), _ptr(b),
                                                 _ptr(h0), _ptr(y), int(threads))
        if rc != 0:
            raise ValueError("oracle_rnn_forward_threads rejected its arguments")
        return y

    def forward_csr(self, x, Wx, row_ptr, cols, vals, b, h0=None) -> np.ndarray:
        """y[T,B,H] for unbalanced sparse Wh in compressed-row form:
        row_ptr[H+1], cols[nnz], vals[nnz]."""
        x, Wx, vals, b = _f64(x), _f64(Wx), _f64(vals), _f64(b)
        row_ptr = np.ascontiguousarray(np.asarray(row_ptr, dtype=np.int64))
        cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        T, B, I = x.shape
        H = Wx.shape[0]
        assert row_ptr.shape == (H + 1,) and cols.shape == vals.shape
        h0 = None if h0 is None else _f64(h0)
        y = np.zeros((T, B, H), dtype=np.float64)
        rc = self.lib.oracle_rnn_forward_csr(T, B, H, I, _ptr(x), _ptr(Wx), _ptr(row_ptr, _L),
                                             _ptr(vals), _ptr(cols, _L), _ptr(b), _ptr(h0),
                                             _ptr(y))
        if rc != 0:
            raise ValueError("oracle_rnn_forward_csr rejected its arguments")
        return y

    def forward_stack(self, x, layers, h0=None) -> np.ndarray:
        """y[L,T,B,H] of a stack of dense layers: layer 0 reads x, layer l > 0
        reads layer l-1's output sequence; layers[l] = (Wx_l, Wh_l, b_l),
        h0[L,B,H] or None.  The definition of stacking written out: each
        layer is the pinned single-layer oracle applied to the layer below's
        output ("Optimizing Performance of Recurrent Neural Networks on
        GPUs", Abstract: multi-layer networks)."""
        ys = []
        inp = x
        for l, (Wx, Wh, b) in enumerate(layers):
            y = self.forward_dense(inp, Wx, Wh, b, None if h0 is None else h0[l])
            ys.append(y)
            inp = y
        return np.stack(ys)

    def forward(self, p, T: Optional[int] = None, threads: int = 1) -> np.ndarray:
        """Run a ``synth.Problem`` (optionally only its first ``T`` steps);
        ``threads`` > 1 runs a single dense or row-balanced layer on that many
        host threads."""
        x = p.x if T is None else p.x[:T]
        if threads > 1:
            assert getattr(p, "layers", None) is None and getattr(p, "row_ptr", None) is None
            if p.sparse:
                return self.forward_threads(x, p.Wx, p.b, p.h0, vals=p.vals, cols=p.cols,
                                            threads=threads)
            return self.forward_threads(x, p.Wx, p.b, p.h0, Wh=p.Wh, threads=threads)
        if getattr(p, "layers", None) is not None:
            return self.forward_stack(x, p.layers, p.h0)
        if getattr(p, "row_ptr", None) is not None:
            return self.forward_csr(x, p.Wx, p.row_ptr, p.cols, p.vals, p.b, p.h0)
        if p.sparse:
            return self.forward_sparse(x, p.Wx, p.vals, p.cols, p.b, p.h0)
        return self.forward_dense(x, p.Wx, p.Wh, p.b, p.h0)

    # -- backward (BPTT) ---------------------------------------------------
    def backward_dense(self, x, Wx, Wh, b, h0, dy) -> dict:
        """Gradients of L = sum(dy * y) for dense Wh: keys delta [T,B,H],
        dx [T,B,I], dh0 [B,H], dWx [H,I], dWh [H,H], db [H] (the C function
        runs its own forward for y)."""
        x, Wx, Wh, b, dy = _f64(x), _f64(Wx), _f64(Wh), _f64(b), _f64(dy)
        T, B, I = x.shape
        H = Wh.shape[0]
        assert dy.shape == (T, B, H) and Wx.shape == (H, I) and Wh.shape == (H, H)
        h0 = None if h0 is None else _f64(h0)
        out = {"delta": np.zeros((T, B, H)), "dx": np.zeros((T, B, I)),
               "dh0": np.zeros((B, H)), "dWx": np.zeros((H, I)), "dWh": np.zeros((H, H)),
               "db": np.zeros(H)}
        rc = self.lib.oracle_rnn_backward_dense(
            T, B, H, I, _ptr(x), _ptr(Wx), _ptr(Wh), _ptr(b), _ptr(h0), _ptr(dy),
            _ptr(out["delta"]), _ptr(out["dx"]), _ptr(out["dh0"]), _ptr(out["dWx"]),
            _ptr(out["dWh"]), _ptr(out["db"]))
        if rc != 0:
            raise ValueError("oracle_rnn_backward_dense rejected its arguments")
        return out

    def backward(self, p, dy) -> dict:
        """Gradients for a ``synth.Problem``.  Sparse weights: the loss depends on
        a stored entry (r, cols[r][j]) only through that position of the
        matrix, so its gradient is dWh[r, cols[r][j]] of the same matrix held
        densely; returned as dvals in the storage order ([H,k], or [nnz] for
        compressed rows) next to the dense dWh."""
        if p.sparse:
            Wh = np.zeros((p.H, p.H))
            if getattr(p, "row_ptr", None) is not None:
                rows = np.repeat(np.arange(p.H), np.diff(p.row_ptr))
                cols = p.cols.astype(np.int64)
                Wh[rows, cols] = p.vals.astype(np.float64)
            else:
                rows = np.repeat(np.arange(p.H), p.k)
                cols = p.cols.astype(np.int64).ravel()
                Wh[rows, cols] = p.vals.astype(np.float64).ravel()
            g = self.backward_dense(p.x, p.Wx, Wh, p.b, p.h0, dy)
            dv = g["dWh"][rows, cols]
            g["dvals"] = dv if getattr(p, "row_ptr", None) is not None else dv.reshape(p.H, p.k)
            return g
        return self.backward_dense(p.x, p.Wx, p.Wh, p.b, p.h0, dy)

    def delta_cells(self, Wh, samples, dy_of, y_of, delta_next_of) -> np.ndarray:
        """Single elements of the reverse recurrence: for each (t, b, r),
        [y_t > 0] * (dy_t[r] + sum_c Wh[c, r] delta_{t+1}[c]) with the three
        vectors supplied by the callbacks (delta_next_of may return None)."""
        Wh = _f64(Wh)
        H = Wh.shape[0]
        out = np.zeros(len(samples))
        for i, (t, bb, r) in enumerate(samples):
            nx = delta_next_of(t, bb)
            out[i] = self.lib.oracle_rnn_delta_cell_dense(
                H, r, _ptr(Wh), _ptr(_f64(dy_of(t, bb))), _ptr(_f64(y_of(t, bb))),
                None if nx is None else _ptr(_f64(nx)))
        return out

    # -- pieces ----------------------------------------------------------
    def input_projection(self, x, Wx, b) -> np.ndarray:
        """P[T,B,H] = Wx x + b for every step."""
        x, Wx, b = _f64(x), _f64(Wx), _f64(b)
        T, B, I = x.shape
        H = Wx.shape[0]
        P = np.zeros((T, B, H), dtype=np.float64)
        rc = self.lib.oracle_rnn_input_projection(T, B, H, I, _ptr(x), _ptr(Wx),
                                                  _ptr(b), _ptr(P))
        if rc != 0:
            raise ValueError("oracle_rnn_input_projection rejected its arguments")
        return P

    def cells(self, p, samples, x_t_of, h_prev_of) -> np.ndarray:
        """Single outputs of single steps: for each (t, b, r) in ``samples``,
        ReLU(b[r] + Wx[r,:] x_t[b] + Wh[r,:] h_prev[b]) with x_t and h_prev
        supplied by the callbacks (the teacher-forced check at full size)."""
        Wx = _f64(p.Wx)
        b = _f64(p.b)
        H, I = Wx.shape
        csr = getattr(p, "row_ptr", None) is not None
        if csr:
            vals = _f64(p.vals)
            cols = np.ascontiguousarray(p.cols.astype(np.int64))
            row_ptr = np.ascontiguousarray(p.row_ptr.astype(np.int64))
        elif p.sparse:
            vals = _f64(p.vals)
            cols = np.ascontiguousarray(p.cols.astype(np.int64))
            k = vals.shape[1]
        else:
            Wh = _f64(p.Wh)
        out = np.zeros(len(samples), dtype=np.float64)
        for i, (t, bb, r) in enumerate(samples):
            x_t = _f64(x_t_of(t, bb))
            h_prev = _f64(h_prev_of(t, bb))
            if csr:
                out[i] = self.lib.oracle_rnn_cell_csr(H, I, r, _ptr(x_t), _ptr(Wx),
                                                      _ptr(row_ptr, _L), _ptr(vals),
                                                      _ptr(cols, _L), _ptr(b), _ptr(h_prev))
            elif p.sparse:
                out[i] = self.lib.oracle_rnn_cell_sparse(H, I, k, r, _ptr(x_t), _ptr(Wx),
                                                         _ptr(vals), _ptr(cols, _L),
                                                         _ptr(b), _ptr(h_prev))
            else:
                out[i] = self.lib.oracle_rnn_cell_dense(H, I, r, _ptr(x_t), _ptr(Wx),
                                                        _ptr(Wh), _ptr(b), _ptr(h_prev))
        return out


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from ``prnn_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
