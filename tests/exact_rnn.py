"""An independent, exact-rational statement of the ReLU RNN forward step, used
only to pin the fp64 oracle on tiny inputs.  Written separately from the C
oracle (Python ``fractions.Fraction``, no floating point), so an indexing or
sign mistake in one is not shared by the other."""
from __future__ import annotations

from fractions import Fraction


def _q(v) -> Fraction:
    return v if isinstance(v, Fraction) else Fraction(float(v))


def forward_exact(x, Wx, Wh, b, h0=None):
    """y as nested lists of Fractions: y[t][b][r]."""
    T, B, I = len(x), len(x[0]) if len(x) else 0, len(Wx[0])
    H = len(Wx)
    Wx = [[_q(v) for v in row] for row in Wx]
    Wh = [[_q(v) for v in row] for row in Wh]
    bias = [_q(v) for v in b]
    h = [[Fraction(0)] * H for _ in range(B)] if h0 is None else \
        [[_q(v) for v in row] for row in h0]
    ys = []
    for t in range(T):
        new_h = []
        for bb in range(B):
            xt = [_q(v) for v in x[t][bb]]
            row_out = []
            for r in range(H):
                pre = bias[r]
                pre += sum((Wx[r][i] * xt[i] for i in range(I)), Fraction(0))
                pre += sum((Wh[r][c] * h[bb][c] for c in range(H)), Fraction(0))
                row_out.append(pre if pre > 0 else Fraction(0))
            new_h.append(row_out)
        h = new_h
        ys.append(new_h)
    return ys


def densify(vals, cols, H):
    """Dense [H][H] rational matrix from row-balanced (value, column) lists."""
    W = [[Fraction(0)] * H for _ in range(H)]
    for r in range(len(vals)):
        for v, c in zip(vals[r], cols[r]):
            W[r][int(c)] += _q(v)
    return W
