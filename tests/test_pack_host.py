"""CPU tests of the host-side sparse packing (no GPU): index handling and row
balancing must be bit-exact, and the bank-aware placement must beat a random
one.  Calls prnn_pack_sparse_host through the C ABI."""
import math

import numpy as np
import pytest

from persistent_rnn_recurrence_gb300 import synth


@pytest.fixture(scope="module")
def prnn():
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    from persistent_rnn_recurrence_gb300 import prnn as m
    return m


def unpack(out, ept):
    n, R, q4, tpr, _ = out.shape
    return out.transpose(0, 1, 3, 2, 4).reshape(n, R, tpr, ept)


CASES = [  # (H, k, tpr) incl. the benchmarked layouts and ragged ones
    (1792, 179, 16), (5760, 57, 8), (5760, 288, 8), (300, 17, 4), (260, 3, 1),
    (132, 12, 2), (4096, 40, 2), (64, 64, 32), (33, 5, 8),
]


@pytest.mark.parametrize("H,k,tpr", CASES)
def test_pack_is_an_exact_permutation_of_each_row(prnn, H, k, tpr):
    p = synth.make_problem(H=H, B=1, T=1, k=k, seed=H + k)
    R = math.ceil(H / 152) if H > 152 else 1
    n = math.ceil(H / R)
    out, ept, cap = prnn.prnn_pack_sparse_host(H, k, n, R, tpr, p.vals, p.cols)
    assert ept % 4 == 0 and ept * tpr >= k and (ept - 4) * tpr < k   # minimal padding
    e = unpack(out, ept)
    vbits = (e & 0xFFFF).astype(np.uint16)
    cols = (e >> 16).astype(np.int64)
    assert cols.max() < H
    for c in range(n):
        for r in range(R):
            g = c * R + r
            flat_v, flat_c = vbits[c, r].ravel(), cols[c, r].ravel()
            if g >= H:
                assert (flat_v == 0).all()
                continue
            want = sorted(zip(p.cols[g].astype(np.int64).tolist(),
                              p.vals[g].view(np.uint16).tolist()))
            pad = flat_v == 0
            nz_want = [w for w in want if w[1] != 0]
            got = sorted(zip(flat_c[~pad].tolist(), flat_v[~pad].tolist()))
            assert got == nz_want, (c, r)
            # every original entry appears exactly once (zero-valued ones among the pads)
            assert len(flat_v) - len(nz_want) >= ept * tpr - k


def test_bank_aware_placement_beats_random(prnn):
    H, k, tpr = 1792, 179, 16
    p = synth.make_problem(H=H, B=1, T=1, k=k, seed=3)
    R, n = 12, 150
    out, ept, cap = prnn.prnn_pack_sparse_host(H, k, n, R, tpr, p.vals, p.cols)
    res = unpack(out, ept) >> 16 & 31
    rng = np.random.default_rng(0)
    waves, rand = [], []
    for c in range(n):
        for w in range(R // 2):
            blk = res[c, 2 * w:2 * w + 2].reshape(32, ept)
            for j in range(ept):
                waves.append(np.bincount(blk[:, j], minlength=32).max())
                rand.append(np.bincount(rng.integers(0, 32, 32), minlength=32).max())
    assert cap <= 4
    assert np.mean(waves) < 0.7 * np.mean(rand)


def test_pack_rejects_bad_indices(prnn):
    p = synth.make_problem(H=64, B=1, T=1, k=8, seed=1)
    bad = p.cols.copy()
    bad[3, 2] = bad[3, 1]
    with pytest.raises(prnn.PrnnError):
        prnn.prnn_pack_sparse_host(64, 8, 64, 1, 8, p.vals, bad)
    bad = p.cols.copy()
    bad[0, 0] = 64
    with pytest.raises(prnn.PrnnError):
        prnn.prnn_pack_sparse_host(64, 8, 64, 1, 8, p.vals, bad)
    with pytest.raises(prnn.PrnnError):                      # threads per row must be 2^j
        prnn.prnn_pack_sparse_host(64, 8, 64, 1, 3, p.vals, p.cols)
    with pytest.raises(prnn.PrnnError):                      # too few rows
        prnn.prnn_pack_sparse_host(64, 8, 10, 1, 8, p.vals, p.cols)
