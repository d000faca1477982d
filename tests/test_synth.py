"""CPU tests of the seeded input generator (shapes, dtypes, row balance,
determinism) -- the generator feeds both the oracle and the CUDA path."""
import numpy as np

from persistent_rnn_recurrence_gb300 import synth


def test_named_shapes_and_dtypes():
    p = synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=4)
    assert p.x.shape == (4, 4, 1792) and p.x.dtype == np.float32
    assert p.Wx.shape == (1792, 1792) and p.Wx.dtype == np.float16
    assert p.vals.shape == (1792, 179) and p.vals.dtype == np.float16
    assert p.cols.dtype == np.uint16 and p.k == 179 and p.h0 is None
    q = synth.named_problem("dense_f32_h256_b4_t32")
    assert q.Wh.dtype == np.float32 and q.Wh.shape == (256, 256) and q.T == 32
    r = synth.named_problem("dense_f16_h1152_b4_t256", T=2)
    assert r.h0.shape == (4, 1152) and r.Wh.dtype == np.float16


def test_row_balanced_columns():
    p = synth.make_problem(H=300, B=2, T=2, k=31, seed=5)
    c = p.cols.astype(np.int64)
    assert c.shape == (300, 31)
    assert (np.diff(c, axis=1) > 0).all()          # ascending and distinct per row
    assert c.min() >= 0 and c.max() < 300


def test_density_to_k():
    assert synth.sparse_k(1792, 0.10) == 179
    assert synth.sparse_k(5760, 0.01) == 57 and synth.sparse_k(5760, 0.05) == 288
    assert [synth.sparse_k(4096, d) for d in (0.25, 0.10, 0.01)] == [1024, 409, 40]


def test_seeded_determinism():
    a = synth.make_problem(H=64, B=2, T=3, k=8, seed=9, h0_std=0.1)
    b = synth.make_problem(H=64, B=2, T=3, k=8, seed=9, h0_std=0.1)
    for f in ("x", "Wx", "vals", "cols", "b", "h0"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_sweep_has_48_points():
    pts = list(synth.sweep_points())
    assert len(pts) == 48 and len({n for n, _ in pts}) == 48
