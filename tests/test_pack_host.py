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


PLACED_CASES = [  # (H, k, tpr, R, n_cta): the benchmarked layouts, full-slot and ragged ones
    (1792, 179, 8, 48, 38), (5760, 57, 8, 152, 38), (5760, 288, 8, 152, 38),
    (2304, 576, 16, 61, 38), (1152, 115, 8, 31, 38), (128, 16, 4, 8, 16), (300, 17, 4, 2, 150),
]


def staged_positions(place, H):
    """Position of every column under one CTA's table, restated from the
    documented rule: column 4g+j goes to 128*(g//32) + 32*j + byte j of place[g]."""
    g = np.arange(H) // 4
    j = np.arange(H) % 4
    byte = (place[g].astype(np.int64) >> (8 * j)) & 0xFF
    return 128 * (g // 32) + 32 * j + byte


@pytest.mark.parametrize("H,k,tpr,R,n", PLACED_CASES)
def test_placed_pack_keeps_rows_and_balances_banks(prnn, H, k, tpr, R, n):
    p = synth.make_problem(H=H, B=1, T=1, k=k, seed=H + 7 * k)
    out, place, ept, cap = prnn.prnn_pack_sparse_host_placed(H, k, n, R, tpr, p.vals, p.cols)
    if H % 128:
        # column order: exactly the unplaced packing
        ref, ept0, cap0 = prnn.prnn_pack_sparse_host(H, k, n, R, tpr, p.vals, p.cols)
        assert place is None and ept == ept0 and np.array_equal(out, ref)
        return
    assert place.shape == (n, H // 4)
    e = unpack(out, ept)
    vbits = (e & 0xFFFF).astype(np.uint16)
    idx = (e >> 16).astype(np.int64)
    rpw = 32 // tpr
    for c in range(n):
        # every class (block of 128 columns, component j) is a permutation of the banks
        for blk in range(H // 128):
            for j in range(4):
                banks = (place[c, 32 * blk:32 * blk + 32].astype(np.int64) >> (8 * j)) & 0xFF
                assert sorted(banks.tolist()) == list(range(32)), (c, blk, j)
        pos = staged_positions(place[c], H)
        assert sorted(pos.tolist()) == list(range(H))
        col_at = np.empty(H, dtype=np.int64)
        col_at[pos] = np.arange(H)
        for r in range(R):
            g = c * R + r
            if g >= H:
                assert (vbits[c, r] == 0).all()
                continue
            fv, fi = vbits[c, r].ravel(), idx[c, r].ravel()
            pad = fv == 0
            want = sorted((cc, v) for cc, v in zip(p.cols[g].astype(np.int64).tolist(),
                                                    p.vals[g].view(np.uint16).tolist()) if v != 0)
            got = sorted(zip(col_at[fi[~pad]].tolist(), fv[~pad].tolist()))
            assert got == want, (c, r)
        # gather slots: the lanes of a warp that own a row use distinct banks
        for w in range((R + rpw - 1) // rpw):
            rows = [r for r in range(w * rpw, min(R, w * rpw + rpw)) if c * R + r < H]
            if not rows:
                continue
            blkidx = idx[c, rows].reshape(len(rows) * tpr, ept)
            worst = max(np.bincount(blkidx[:, s] % 32, minlength=32).max() for s in range(ept))
            assert worst <= cap
    if (H, k) in ((1792, 179), (5760, 57), (5760, 288), (2304, 576)):
        assert cap == 1


def test_placed_pack_reproduces_the_product(prnn):
    """Emulates one step of the kernel on the CPU: stage h by the documented
    placement rule, gather every packed entry at its index, sum per row, and
    compare with Wh @ h from the unpacked rows."""
    H, k, tpr, R, n = 1792, 179, 8, 48, 38
    p = synth.make_problem(H=H, B=1, T=1, k=k, seed=11)
    out, place, ept, cap = prnn.prnn_pack_sparse_host_placed(H, k, n, R, tpr, p.vals, p.cols)
    h = np.random.default_rng(5).standard_normal(H)
    want = np.array([np.dot(p.vals[r].astype(np.float64), h[p.cols[r].astype(np.int64)])
                     for r in range(H)])
    e = unpack(out, ept)
    got = np.zeros(H)
    for c in range(n):
        hs = np.full(H, np.nan)
        hs[staged_positions(place[c], H)] = h
        assert not np.isnan(hs).any()
        vals = (e[c] & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
        prod = vals * hs[(e[c] >> 16).astype(np.int64)]
        rows = min(R, H - c * R)
        got[c * R:c * R + rows] = prod[:rows].reshape(rows, -1).sum(1)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_placed_pack_is_deterministic(prnn):
    """The placement search is seeded: packing the same weights twice gives
    the same tables and the same packed words."""
    H, k, tpr, R, n = 1152, 115, 8, 31, 38
    p = synth.make_problem(H=H, B=1, T=1, k=k, seed=12)
    a = prnn.prnn_pack_sparse_host_placed(H, k, n, R, tpr, p.vals, p.cols)
    b = prnn.prnn_pack_sparse_host_placed(H, k, n, R, tpr, p.vals, p.cols)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2:] == b[2:]
    # CTAs get different orders (each balances its own warps)
    assert not np.array_equal(a[1][0], a[1][1])


def _random_layouts(n):
    rng = np.random.default_rng(2024)
    out = []
    while len(out) < n:
        H = int(rng.choice([128, 256, 384, 40, 97, 130]))
        tpr = int(rng.choice([1, 2, 4, 8, 16, 32]))
        k = int(rng.choice([1, 2, 3, max(1, H // 10), H // 2, H]))
        R = int(rng.integers(1, 9))
        n_cta = -(-H // R)
        out.append((H, k, tpr, R, n_cta, int(rng.integers(1 << 30))))
    return out


@pytest.mark.parametrize("H,k,tpr,R,n,seed", _random_layouts(24))
def test_random_layouts_pack_exactly(prnn, H, k, tpr, R, n, seed):
    """Both packings on random small layouts (k = 1 .. H, every threads-per-row,
    ragged row counts): every row keeps exactly its (column, value) entries,
    padding is zero-valued, indices stay on the staged h, and no gather slot
    puts more lanes on a bank than the reported cap."""
    rng = np.random.default_rng(seed)
    cols = np.stack([np.sort(rng.choice(H, k, replace=False)) for _ in range(H)]).astype(np.uint16)
    vals = rng.standard_normal((H, k)).astype(np.float16)
    vals[vals == 0] = np.float16(0.5)          # keep every real entry non-zero
    for placed in (False, True):
        if placed:
            out, place, ept, cap = prnn.prnn_pack_sparse_host_placed(H, k, n, R, tpr, vals, cols)
            col_of = []
            for c in range(n):
                if place is None:
                    col_of.append(np.arange(H))
                else:
                    pos = staged_positions(place[c], H)
                    inv = np.empty(H, dtype=np.int64)
                    inv[pos] = np.arange(H)
                    col_of.append(inv)
        else:
            out, ept, cap = prnn.prnn_pack_sparse_host(H, k, n, R, tpr, vals, cols)
            col_of = [np.arange(H)] * n
        e = unpack(out, ept)
        v = (e & 0xFFFF).astype(np.uint16)
        idx = (e >> 16).astype(np.int64)
        assert idx.max() < H
        rpw = max(1, 32 // tpr)
        for c in range(n):
            for r in range(R):
                g = c * R + r
                if g >= H:
                    continue
                fv, fi = v[c, r].ravel(), idx[c, r].ravel()
                real = fv != 0
                got = sorted(zip(col_of[c][fi[real]].tolist(), fv[real].tolist()))
                want = sorted(zip(cols[g].astype(np.int64).tolist(), vals[g].view(np.uint16).tolist()))
                assert got == want, (placed, c, r)
            for w in range(-(-R // rpw)):
                rows = [r for r in range(w * rpw, min(R, w * rpw + rpw)) if c * R + r < H]
                if not rows:
                    continue
                lanes = idx[c, rows].reshape(len(rows) * tpr, ept)
                for j in range(ept):
                    # wavefronts of this slot: the most distinct addresses on one bank
                    # (lanes reading the same word share it)
                    addrs = np.unique(lanes[:, j])
                    assert np.bincount(addrs % 32, minlength=32).max() <= max(cap, 1), \
                        (placed, c, w, j)


# ---- the tensor-core K-split kernel's weight image (prnn_pack_dense_ksplit_host) ----

KSPLIT_CASES = [(128, 2), (128, 8), (384, 7), (640, 8), (1152, 8), (1152, 5), (2304, 6), (4096, 4)]


def _unswizzle(img):
    """[nblk, cs, nat, 128, 64] -> [nblk, cs, 128, nat * 64]: each row's
    16-byte chunk p holds logical chunk p XOR (row mod 8) (the 128-byte
    swizzle), atoms of one slice side by side in K."""
    m = np.arange(128)[:, None]
    L = np.arange(64)[None, :]
    idx = ((L // 8) ^ (m % 8)) * 8 + L % 8                      # [128, 64]
    u = np.take_along_axis(img, np.broadcast_to(idx, img.shape), axis=-1)
    nblk, cs, nat = img.shape[:3]
    return u.transpose(0, 1, 3, 2, 4).reshape(nblk, cs, 128, nat * 64)


@pytest.mark.parametrize("H,cs", KSPLIT_CASES)
def test_ksplit_image_places_every_weight_once(prnn, H, cs):
    r, c = np.meshgrid(np.arange(H), np.arange(H), indexing="ij")
    rows = prnn.prnn_pack_dense_ksplit_host(H, cs, (r + 1).astype(np.uint16))
    cols = _unswizzle(prnn.prnn_pack_dense_ksplit_host(H, cs, (c + 1).astype(np.uint16)))
    rows = _unswizzle(rows)
    nblk, cs_, _, width = cols.shape
    assert (nblk, cs_) == (H // 128, cs)
    # slice widths: whole 16-column steps, as even as possible, tiling 0 .. H-1
    kl = [(cols[0, j, 0] != 0).sum() for j in range(cs)]
    assert sum(kl) == H and all(w % 16 == 0 for w in kl) and max(kl) - min(kl) <= 16
    assert width == -(-max(kl) // 64) * 64                     # whole atoms, no spare one
    k0 = np.concatenate([[0], np.cumsum(kl)[:-1]])
    for j in range(cs):
        w = kl[j]
        # every row of the slice holds columns k0 .. k0 + kl - 1 in order, then zeros
        assert (cols[:, j, :, :w] == (k0[j] + np.arange(w) + 1)[None, None, :]).all()
        assert (cols[:, j, :, w:] == 0).all() and (rows[:, j, :, w:] == 0).all()
        # lane m of block bk is row 128 bk + m of Wh
        want_r = (np.arange(nblk)[:, None] * 128 + np.arange(128)[None, :] + 1)
        assert (rows[:, j, :, :w] == want_r[:, :, None]).all()


@pytest.mark.parametrize("H,cs", [(256, 3), (640, 8)])
def test_ksplit_transposed_image_is_the_image_of_the_transpose(prnn, H, cs):
    rng = np.random.default_rng(H + cs)
    w = rng.normal(size=(H, H)).astype(np.float16)
    a = prnn.prnn_pack_dense_ksplit_host(H, cs, w, transpose=True)
    b = prnn.prnn_pack_dense_ksplit_host(H, cs, np.ascontiguousarray(w.T))
    assert np.array_equal(a, b)
    assert not np.array_equal(a, prnn.prnn_pack_dense_ksplit_host(H, cs, w))


def test_ksplit_image_errors(prnn):
    w = np.zeros((256, 256), dtype=np.float16)
    for H, cs in ((256, 1), (256, 9)):
        with pytest.raises(prnn.PrnnError):
            prnn.prnn_pack_dense_ksplit_host(H, cs, w)
    with pytest.raises(prnn.PrnnError):                         # not a multiple of 128
        prnn.prnn_pack_dense_ksplit_host(200, 2, np.zeros((200, 200), dtype=np.float16))
    with pytest.raises(prnn.PrnnError):                         # 128 / 16 = 8 steps < 9 slices
        prnn.prnn_pack_dense_ksplit_host(128, 9, np.zeros((128, 128), dtype=np.float16))
    import ctypes
    need = ctypes.c_size_t()
    small = np.zeros(10, dtype=np.uint16)
    st = prnn._lib.prnn_pack_dense_ksplit_host(256, 2, w.ctypes.data, 0, small.ctypes.data,
                                              small.size, ctypes.byref(need))
    assert st == prnn.PRNN_ERR_INVALID_ARG and need.value == 2 * 2 * 2 * 8192
    assert (small == 0).all()                                   # nothing written


@pytest.mark.parametrize("H,cs", [(384, 7), (1152, 8)])
def test_ksplit_image_matches_the_header_formula(prnn, H, cs):
    """The element placement include/prnn.h documents for
    prnn_pack_dense_ksplit_host, evaluated for every weight."""
    rng = np.random.default_rng(7 * H + cs)
    w = rng.integers(1, 1 << 15, size=(H, H), dtype=np.uint16)  # no zero weights
    flat = prnn.prnn_pack_dense_ksplit_host(H, cs, w).ravel()
    steps = H // 16
    k0 = [16 * (j * steps // cs) for j in range(cs + 1)]
    nat = -(-(-(-steps // cs)) // 4)
    assert flat.size == (H // 128) * cs * nat * 8192
    r, c = np.meshgrid(np.arange(H), np.arange(H), indexing="ij")
    j = np.searchsorted(np.array(k0), c, side="right") - 1
    kc = c - np.array(k0)[j]
    bk, m = r // 128, r % 128
    pos = ((bk * cs + j) * nat + kc // 64) * 8192 + m * 64 + (((kc % 64) // 8) ^ (m % 8)) * 8 + kc % 8
    assert np.array_equal(flat[pos], w)
    rest = np.ones(flat.size, dtype=bool)
    rest[pos.ravel()] = False
    assert (flat[rest] == 0).all()
