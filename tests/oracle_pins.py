"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:
  * the hand-worked integer example in tests/golden/ (literal values),
  * closed forms: Wh = 0 gives y_t = ReLU(Wx x_t + b); T = 1 gives
    y_0 = ReLU(Wx x_0 + Wh h0 + b) (numpy matrix products, a different code path),
  * the linear regime: with non-negative integer data ReLU is the identity, so
    h_t = Wh^{t+1} h0 + sum_{j<=t} Wh^{t-j} (Wx x_j + b) exactly (Python ints),
  * exact rational brute force on tiny sizes (tests/exact_rnn.py),
  * positive homogeneity (x, b, h0 scaled by 2 scale y by exactly 2),
  * sparse form equals the densified dense form bit for bit,
  * chaining and batch independence (the recurrence's own structure).
The mutation test runs all of them against deliberately broken oracle builds
and requires each mistake to trip at least one pin.
"""
from __future__ import annotations

import json
import os

import numpy as np

from tests.exact_rnn import densify, forward_exact

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _relu(a):
    return np.where(a > 0, a, 0.0)


def _rand(rng, *shape, scale=1.0):
    return rng.normal(0.0, scale, size=shape)


def _dyadic(rng, *shape, denom=8, lo=-12, hi=12):
    """Small multiples of 1/denom: exact in fp16, fp64 and Fraction."""
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) / denom


def pin_hand_computed(o):
    g = json.load(open(os.path.join(GOLDEN, "hand_h2_i2_b2_t3.json")))
    y = o.forward_dense(np.array(g["x"], float), np.array(g["Wx"], float),
                        np.array(g["Wh"], float), np.array(g["b"], float),
                        np.array(g["h0"], float))
    assert np.array_equal(y, np.array(g["y"], float)), y


def pin_hand_computed_sparse(o):
    """The same worked example with Wh given as 2 (value, column) pairs per row,
    columns deliberately listed out of order in row 1."""
    g = json.load(open(os.path.join(GOLDEN, "hand_h2_i2_b2_t3.json")))
    Wh = np.array(g["Wh"], float)
    vals = np.array([[Wh[0, 0], Wh[0, 1]], [Wh[1, 1], Wh[1, 0]]])
    cols = np.array([[0, 1], [1, 0]])
    y = o.forward_sparse(np.array(g["x"], float), np.array(g["Wx"], float), vals, cols,
                         np.array(g["b"], float), np.array(g["h0"], float))
    assert np.array_equal(y, np.array(g["y"], float)), y


def pin_wh_zero_identity(o):
    rng = np.random.default_rng(11)
    T, B, H, I = 4, 3, 7, 5
    x, Wx, b = _rand(rng, T, B, I), _rand(rng, H, I), _rand(rng, H)
    h0 = _rand(rng, B, H)
    y = o.forward_dense(x, Wx, np.zeros((H, H)), b, h0)
    ref = _relu(np.einsum("tbi,ri->tbr", x, Wx) + b)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13), np.abs(y - ref).max()
    # the projection alone is the pre-activation of the same closed form
    P = o.input_projection(x, Wx, b)
    assert np.allclose(P, np.einsum("tbi,ri->tbr", x, Wx) + b, rtol=1e-13, atol=1e-13)


def pin_t1_closed_form(o):
    rng = np.random.default_rng(12)
    B, H, I = 3, 6, 9
    x, Wx, Wh, b = _rand(rng, 1, B, I), _rand(rng, H, I), _rand(rng, H, H), _rand(rng, H)
    h0 = _rand(rng, B, H)
    y = o.forward_dense(x, Wx, Wh, b, h0)
    ref = _relu(x[0] @ Wx.T + h0 @ Wh.T + b)
    assert np.allclose(y[0], ref, rtol=1e-13, atol=1e-13), np.abs(y[0] - ref).max()
    # h0 = NULL means zeros
    y0 = o.forward_dense(x, Wx, Wh, b, None)
    assert np.allclose(y0[0], _relu(x[0] @ Wx.T + b), rtol=1e-13, atol=1e-13)


def pin_linear_regime_exact(o):
    """Non-negative integers: every pre-activation is >= 0, ReLU is the
    identity, and the recurrence is a linear system with an exact
    matrix-power solution (computed with Python integers)."""
    rng = np.random.default_rng(13)
    T, B, H, I = 5, 2, 3, 2
    x = rng.integers(0, 3, size=(T, B, I))
    Wx = rng.integers(0, 3, size=(H, I))
    Wh = rng.integers(0, 2, size=(H, H))
    Wh[0, 2] = 1
    Wh[2, 0] = 0                       # make Wh asymmetric
    b = rng.integers(0, 3, size=H)
    h0 = rng.integers(0, 3, size=(B, H))
    y = o.forward_dense(x, Wx, Wh, b, h0)
    Whi = [[int(v) for v in row] for row in Wh]

    def matvec(M, v):
        return [sum(M[r][c] * v[c] for c in range(len(v))) for r in range(len(M))]

    for bb in range(B):
        for t in range(T):
            acc = [int(v) for v in h0[bb]]
            for _ in range(t + 1):
                acc = matvec(Whi, acc)                    # Wh^{t+1} h0
            for j in range(t + 1):
                u = [int(b[r]) + sum(int(Wx[r][i]) * int(x[j][bb][i]) for i in range(I))
                     for r in range(H)]
                for _ in range(t - j):
                    u = matvec(Whi, u)                    # Wh^{t-j} (Wx x_j + b)
                acc = [a + c for a, c in zip(acc, u)]
            assert [float(v) for v in acc] == list(y[t, bb]), (t, bb, acc, y[t, bb])


def pin_exact_rational(o):
    rng = np.random.default_rng(14)
    for (T, B, H, I) in [(4, 2, 4, 3), (3, 1, 2, 4), (4, 3, 3, 3)]:
        x = _dyadic(rng, T, B, I)
        Wx, Wh = _dyadic(rng, H, I), _dyadic(rng, H, H)
        b, h0 = _dyadic(rng, H), _dyadic(rng, B, H)
        y = o.forward_dense(x, Wx, Wh, b, h0)
        ref = forward_exact(x.tolist(), Wx.tolist(), Wh.tolist(), b.tolist(), h0.tolist())
        for t in range(T):
            for bb in range(B):
                for r in range(H):
                    assert y[t, bb, r] == float(ref[t][bb][r]), (T, B, H, I, t, bb, r)
    # sparse: rational brute force on the densified matrix
    H, k, T, B = 4, 2, 4, 2
    cols = np.array([[3, 1], [0, 2], [2, 3], [1, 0]])
    vals = _dyadic(rng, H, k)
    x, Wx, b = _dyadic(rng, T, B, H), _dyadic(rng, H, H), _dyadic(rng, H)
    y = o.forward_sparse(x, Wx, vals, cols, b, None)
    W = densify(vals.tolist(), cols.tolist(), H)
    ref = forward_exact(x.tolist(), Wx.tolist(), [[float(v) for v in r] for r in W],
                        b.tolist(), None)
    for t in range(T):
        for bb in range(B):
            assert list(y[t, bb]) == [float(v) for v in ref[t][bb]], (t, bb)


def pin_homogeneity(o):
    rng = np.random.default_rng(15)
    T, B, H, I = 6, 2, 8, 5
    x, Wx, Wh, b = _rand(rng, T, B, I), _rand(rng, H, I), _rand(rng, H, H, scale=0.3), \
        _rand(rng, H)
    h0 = _rand(rng, B, H)
    y1 = o.forward_dense(x, Wx, Wh, b, h0)
    y2 = o.forward_dense(2 * x, Wx, Wh, 2 * b, 2 * h0)
    assert np.array_equal(y2, 2 * y1)
    assert (y1 > 0).any() and (y1 == 0).any()      # both ReLU branches taken


def pin_sparse_equals_densified(o):
    rng = np.random.default_rng(16)
    T, B, H, I, k = 5, 3, 33, 20, 5
    cols = np.stack([np.sort(rng.choice(H, k, replace=False)) for _ in range(H)])
    vals = _rand(rng, H, k, scale=0.5)
    Wh = np.zeros((H, H))
    for r in range(H):
        Wh[r, cols[r]] = vals[r]
    x, Wx, b, h0 = _rand(rng, T, B, I), _rand(rng, H, I), _rand(rng, H), _rand(rng, B, H)
    ys = o.forward_sparse(x, Wx, vals, cols, b, h0)
    yd = o.forward_dense(x, Wx, Wh, b, h0)
    assert np.array_equal(ys, yd)


def pin_csr_equals_densified_and_balanced(o):
    """Unbalanced compressed rows (some empty, some full): bit-identical to
    the dense form of the same matrix (entries sorted by column), and to the
    row-balanced form when every row has the same length."""
    rng = np.random.default_rng(19)
    T, B, H, I = 4, 2, 9, 6
    lens = np.array([0, 9, 3, 1, 5, 2, 7, 4, 3])
    row_ptr = np.concatenate([[0], np.cumsum(lens)])
    cols = np.concatenate([np.sort(rng.choice(H, n, replace=False)) for n in lens])
    vals = _rand(rng, int(lens.sum()), scale=0.4)
    x, Wx, b, h0 = _rand(rng, T, B, I), _rand(rng, H, I), _rand(rng, H), _rand(rng, B, H)
    Wh = np.zeros((H, H))
    for r in range(H):
        Wh[r, cols[row_ptr[r]:row_ptr[r + 1]]] = vals[row_ptr[r]:row_ptr[r + 1]]
    assert np.array_equal(o.forward_csr(x, Wx, row_ptr, cols, vals, b, h0),
                          o.forward_dense(x, Wx, Wh, b, h0))
    k = 3
    bc = np.stack([np.sort(rng.choice(H, k, replace=False)) for _ in range(H)])
    bv = _rand(rng, H, k, scale=0.4)
    assert np.array_equal(o.forward_csr(x, Wx, np.arange(H + 1) * k, bc.ravel(), bv.ravel(), b),
                          o.forward_sparse(x, Wx, bv, bc, b))


def pin_stack_definition(o):
    """Stacked layers: (1) one layer is the single-layer oracle; (2) a top
    layer with Wx = identity, Wh = 0, b = 0 reproduces the layer below exactly
    (ReLU of a non-negative sequence is itself), which a top layer reading x
    instead of the layer below, or taking another layer's h0, breaks; (3) two
    layers of dyadic data with distinct h0 per layer equal exact rational
    brute force applied layer on layer."""
    rng = np.random.default_rng(20)
    T, B, H, I = 4, 2, 5, 3
    x = _rand(rng, T, B, I)
    Wx0, Wh0, b0 = _rand(rng, H, I), _rand(rng, H, H, scale=0.4), _rand(rng, H)
    h0 = _rand(rng, 2, B, H)
    y1 = o.forward_stack(x, [(Wx0, Wh0, b0)], h0[:1])
    assert y1.shape == (1, T, B, H)
    assert np.array_equal(y1[0], o.forward_dense(x, Wx0, Wh0, b0, h0[0]))
    ident = (np.eye(H), np.zeros((H, H)), np.zeros(H))
    y2 = o.forward_stack(x, [(Wx0, Wh0, b0), ident], np.stack([h0[0], 5.0 + h0[1]]))
    assert np.array_equal(y2[1], y2[0]) and (y2[0] > 0).any()
    # exact rational, two layers
    xd = _dyadic(rng, T, B, I)
    L0 = (_dyadic(rng, H, I), _dyadic(rng, H, H), _dyadic(rng, H))
    L1 = (_dyadic(rng, H, H), _dyadic(rng, H, H), _dyadic(rng, H))
    hd = _dyadic(rng, 2, B, H)
    y = o.forward_stack(xd, [L0, L1], hd)
    r0 = forward_exact(xd.tolist(), L0[0].tolist(), L0[1].tolist(), L0[2].tolist(), hd[0].tolist())
    assert y[0].tolist() == [[[float(v) for v in row] for row in step] for step in r0]
    r1 = forward_exact(y[0].tolist(), L1[0].tolist(), L1[1].tolist(), L1[2].tolist(),
                       hd[1].tolist())
    assert y[1].tolist() == [[[float(v) for v in row] for row in step] for step in r1]
    assert (y[1] > 0).any() and (y[1] == 0).any()


def _exact_loss(x, Wx, Wh, b, h0, dy):
    """L = sum(dy * y) in exact rationals (tests/exact_rnn.py)."""
    from fractions import Fraction
    y = forward_exact(x, Wx, Wh, b, h0)
    return sum((Fraction(float(dy[t][bb][r])) * y[t][bb][r]
                for t in range(len(y)) for bb in range(len(y[0])) for r in range(len(y[0][0]))),
               Fraction(0))


def _preacts_nonzero(x, Wx, Wh, b, h0):
    """True when no pre-activation of the exact forward is exactly 0 (the
    loss is then differentiable at this point)."""
    from fractions import Fraction
    T, B, H, I = len(x), len(x[0]), len(Wx), len(Wx[0])
    q = lambda v: Fraction(float(v))
    h = [[Fraction(0)] * H for _ in range(B)] if h0 is None else [[q(v) for v in row] for row in h0]
    for t in range(T):
        nh = []
        for bb in range(B):
            row = []
            for r in range(H):
                a = q(b[r]) + sum(q(Wx[r][i]) * q(x[t][bb][i]) for i in range(I)) + \
                    sum(q(Wh[r][c]) * h[bb][c] for c in range(H))
                if a == 0:
                    return False
                row.append(a if a > 0 else Fraction(0))
            nh.append(row)
        h = nh
    return True


def pin_backward_finite_differences(o):
    """Every gradient of L = sum(dy * y) against exact central differences:
    the loss is evaluated in exact rationals at theta +- eps with
    eps = 1e-30 (the loss is piecewise polynomial in each parameter, so the
    difference quotient is exact up to O(eps^2)), at points with no zero
    pre-activation.  Covers dWh, dWx, db, dh0 and dx, both ReLU branches."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    eps = Fraction(1, 10 ** 30)
    for (T, B, H, I) in [(3, 2, 3, 2), (2, 1, 4, 3)]:
        while True:
            x, Wx, Wh = _dyadic(rng, T, B, I), _dyadic(rng, H, I), _dyadic(rng, H, H, lo=-6, hi=6)
            b, h0, dy = _dyadic(rng, H), _dyadic(rng, B, H), _dyadic(rng, T, B, H)
            if _preacts_nonzero(x.tolist(), Wx.tolist(), Wh.tolist(), b.tolist(), h0.tolist()):
                break
        g = o.backward_dense(x, Wx, Wh, b, h0, dy)
        y = o.forward_dense(x, Wx, Wh, b, h0)
        assert (y > 0).any() and (y == 0).any()
        params = {"Wx": (Wx, "dWx"), "Wh": (Wh, "dWh"), "b": (b, "db"), "h0": (h0, "dh0"),
                  "x": (x, "dx")}
        for name, (arr, gname) in params.items():
            for idx in np.ndindex(arr.shape):
                vals = {}
                for sgn in (1, -1):
                    args = {"x": x.tolist(), "Wx": Wx.tolist(), "Wh": Wh.tolist(),
                            "b": b.tolist(), "h0": h0.tolist()}
                    a = args[name]
                    ref = a
                    for k in idx[:-1]:
                        ref = ref[k]
                    ref[idx[-1]] = Fraction(float(ref[idx[-1]])) + sgn * eps
                    vals[sgn] = _exact_loss(args["x"], args["Wx"], args["Wh"], args["b"],
                                            args["h0"], dy.tolist())
                fd = float((vals[1] - vals[-1]) / (2 * eps))
                got = g[gname][idx]
                assert abs(got - fd) <= 1e-12 * max(1.0, abs(fd)), (name, idx, got, fd)


def pin_backward_linear_regime(o):
    """Non-negative integers keep every unit active, so the reverse
    recurrence is linear: delta_t = sum_{s>=t} (Wh^T)^{s-t} dy_s exactly
    (Python integers), and db = sum over t, b of delta_t."""
    rng = np.random.default_rng(22)
    T, B, H, I = 4, 2, 3, 2
    x = rng.integers(0, 3, size=(T, B, I))
    Wx = rng.integers(1, 3, size=(H, I))
    Wh = rng.integers(0, 2, size=(H, H))
    Wh[0, 1], Wh[1, 0] = 1, 0
    b = rng.integers(1, 3, size=H)
    dy = rng.integers(-3, 4, size=(T, B, H))
    g = o.backward_dense(x, Wx, Wh, b, None, dy)
    WT = [[int(Wh[c][r]) for c in range(H)] for r in range(H)]
    for bb in range(B):
        for t in range(T):
            acc = [0] * H
            for s in range(t, T):
                v = [int(u) for u in dy[s][bb]]
                for _ in range(s - t):
                    v = [sum(WT[r][c] * v[c] for c in range(H)) for r in range(H)]
                acc = [p + q for p, q in zip(acc, v)]
            assert [float(v) for v in acc] == list(g["delta"][t, bb]), (t, bb)
    assert np.array_equal(g["db"], g["delta"].sum(axis=(0, 1)))


def pin_backward_sparse_is_dense_gather(o):
    """Sparse gradients: dvals[r][j] equals the dense gradient at
    (r, cols[r][j]), and perturbing one stored value changes the loss at
    that rate (fp64 central difference, eps = 1e-6, well inside every
    ReLU branch for this draw)."""
    from persistent_rnn_recurrence_gb300 import synth
    p = synth.make_problem(H=12, B=2, T=4, k=3, seed=23, h0_std=0.5)
    rng = np.random.default_rng(24)
    dy = rng.normal(size=(p.T, p.B, p.H))
    g = o.backward(p, dy)
    for r in (0, 5, 11):
        for j in range(p.k):
            c = int(p.cols[r, j])
            assert g["dvals"][r, j] == g["dWh"][r, c]
            base = p.vals.astype(np.float64)
            lo, hi = base.copy(), base.copy()
            lo[r, j] -= 1e-6
            hi[r, j] += 1e-6
            f = lambda v: float((o.forward_sparse(p.x, p.Wx, v, p.cols, p.b, p.h0) * dy).sum())
            fd = (f(hi) - f(lo)) / 2e-6
            assert abs(fd - g["dvals"][r, j]) <= 1e-6 * max(1.0, abs(fd)), (r, j, fd)


def pin_chaining(o):
    rng = np.random.default_rng(17)
    T1, T2, B, H, I = 3, 4, 2, 9, 9
    x, Wx, Wh, b = _rand(rng, T1 + T2, B, I), _rand(rng, H, I), \
        _rand(rng, H, H, scale=0.3), _rand(rng, H)
    h0 = _rand(rng, B, H)
    y = o.forward_dense(x, Wx, Wh, b, h0)
    ya = o.forward_dense(x[:T1], Wx, Wh, b, h0)
    yb = o.forward_dense(x[T1:], Wx, Wh, b, ya[-1])
    assert np.array_equal(y, np.concatenate([ya, yb]))


def pin_batch_independence(o):
    rng = np.random.default_rng(18)
    T, B, H, I = 4, 3, 10, 6
    x, Wx, Wh, b = _rand(rng, T, B, I), _rand(rng, H, I), _rand(rng, H, H, scale=0.3), \
        _rand(rng, H)
    h0 = _rand(rng, B, H)
    y = o.forward_dense(x, Wx, Wh, b, h0)
    for bb in range(B):
        yi = o.forward_dense(x[:, bb:bb + 1], Wx, Wh, b, h0[bb:bb + 1])
        assert np.array_equal(yi[:, 0], y[:, bb])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(o):
    for pin in ALL_PINS:
        pin(o)
