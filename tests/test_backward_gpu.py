"""GPU parity of the backward pass (prnn_backward) against the fp64 oracle.

Three kinds of check:
  * exact-arithmetic problems (dyadic values with few non-zeros per row of
    Wh, so every fp32 sum on the GPU is exact): the GPU forward output equals
    the oracle's bit for bit, so both sides take the same ReLU mask decisions,
    and every gradient must match the oracle's within 1e-6 of its scale;
  * random fp32-weight problems whose pre-activations all stay further from 0
    than the fp32 rounding of the forward (checked on the oracle's side), so
    the masks agree again: every gradient within 1e-4 of its scale;
  * fp16-weight problems on the default path (tensor-core projection and
    bf16 tensor-core gradient products): dyadic problems again, every
    gradient against the oracle's, the bf16 products within their rounding
    bound;
  * fp16-weight and full-size problems, where forward rounding can flip the
    mask of pre-activations near 0: properties that hold at any size --
    every sampled delta equals one oracle step of the reverse recurrence
    applied to the GPU's own y and delta_{t+1} (teacher forcing), and every
    gradient equals its batched product (fp64 numpy) of the GPU's deltas.
"""
import numpy as np
import pytest

import oracle
from persistent_rnn_recurrence_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    from persistent_rnn_recurrence_gb300 import prnn
    return torch, prnn, oracle.default()


def run(env, p, dy, options=None, pre_options=None):
    """pre_options are set before the weights (options that act at set_weights)."""
    torch, prnn, _ = env
    if pre_options:
        lay = prnn.Layer(p.H, p.I, max(1, p.B), p.wdtype, "persistent")
        for k, v in pre_options.items():
            lay.set_option(k, v)
        lay.set_problem_weights(p)
    else:
        lay = prnn.Layer.from_problem(p)
    try:
        for k, v in (options or {}).items():
            lay.set_option(k, v)
        x = torch.from_numpy(p.x).cuda()
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        g = lay.backward(x, y, torch.from_numpy(dy).cuda(), h0)
        assert lay.status() == prnn.PRNN_OK
        return y.cpu().numpy().astype(np.float64), {k: v.cpu().numpy().astype(np.float64)
                                                    for k, v in g.items()}
    finally:
        lay.close()


def rel_err(a, b):
    return float(np.abs(a - b).max()) / max(float(np.abs(b).max()), 1e-30)


def dyadic_problem(seed, H, I, B, T, wdtype, nnz_row=3):
    rng = np.random.default_rng(seed)
    q = lambda *s, lo=-8, hi=8: rng.integers(lo, hi + 1, size=s).astype(np.float64) / 8
    Wh = np.zeros((H, H))
    for r in range(H):
        Wh[r, rng.choice(H, nnz_row, replace=False)] = rng.choice([-0.5, 0.5], nnz_row)
    wt = np.float16 if wdtype == "f16" else np.float32
    p = synth.Problem(name="dyadic", T=T, B=B, H=H, I=I, wdtype=wdtype,
                      x=q(T, B, I).astype(np.float32), Wx=(q(H, I) / 4).astype(wt),
                      b=q(H).astype(np.float32), h0=q(B, H).astype(np.float32), Wh=Wh.astype(wt))
    dy = q(T, B, H)
    return p, dy


@pytest.mark.parametrize("sparse", [False, True])
@pytest.mark.parametrize("shape", [dict(H=1152, I=1152, B=4, T=6), dict(H=640, I=320, B=8, T=5)])
def test_tensor_core_gradients_against_oracle(env, sparse, shape):
    """fp16-weight layers on the default path: tcgen05 projection (x rounded
    to fp16) and tensor-core gradient products from bf16-rounded operands.
    On dyadic problems the forward is exact on both sides (fp16 holds every
    x and weight, fp32 every sum), so the GPU and the oracle take the same
    ReLU decisions: delta, db and dh0 (fp32 arithmetic) must match the
    oracle's gradients within 1e-6, and dWh (or the stored values' gradients),
    dWx and dx -- the bf16 products -- within BF16_PRODUCT_TOL."""
    o = env[2]
    if sparse:
        p, dy = dyadic_sparse_problem(900 + shape["H"], k=3, **shape)
    else:
        p, dy = dyadic_problem(910 + shape["H"], wdtype="f16", **shape)
    y, g = run(env, p, dy.astype(np.float32))
    assert np.array_equal(y, o.forward(p)), "forward not exact: masks could differ"
    assert np.count_nonzero(y) > y.size // 4
    ref = o.backward(p, dy)
    errs = {}
    for k in ("delta", "db", "dh0"):
        errs[k] = rel_err(g[k], ref[k])
        assert errs[k] <= 1e-6, (k, errs[k])
    for k in ("dWx", "dx", "dWh"):
        want = ref["dvals"].ravel() if (sparse and k == "dWh") else ref[k]
        errs[k] = rel_err(g[k].ravel() if sparse and k == "dWh" else g[k], want)
        assert errs[k] <= BF16_PRODUCT_TOL, (k, errs[k])
    print("relative errors vs the oracle:", {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("wdtype", ["f32", "f16"])
@pytest.mark.parametrize("shape", [dict(H=64, I=32, B=3, T=6), dict(H=300, I=100, B=5, T=5),
                                   dict(H=1152, I=1152, B=4, T=4)])
def test_backward_exact_problems(env, wdtype, shape):
    p, dy = dyadic_problem(500 + shape["H"], wdtype=wdtype, **shape)
    o = env[2]
    prnn = env[1]
    # fp32 CUDA-core products everywhere, so every sum stays exact
    y, g = run(env, p, dy.astype(np.float32), {prnn.PRNN_OPT_PROJECTION: 1})
    assert np.array_equal(y, o.forward(p)), "forward not exact: masks could differ"
    ref = o.backward(p, dy)
    for k in ("delta", "dx", "dh0", "dWx", "dWh", "db"):
        assert rel_err(g[k], ref[k]) <= 1e-6, (k, rel_err(g[k], ref[k]))


def _min_abs_preact(o, p):
    y = o.forward(p)
    P = o.input_projection(p.x, p.Wx, p.b)
    h0 = np.zeros((p.B, p.H)) if p.h0 is None else p.h0.astype(np.float64)
    prev = np.concatenate([h0[None], y[:-1]], axis=0)
    a = P + np.einsum("tbc,rc->tbr", prev, p.Wh.astype(np.float64))
    return float(np.abs(a).min())


@pytest.mark.parametrize("shape", [dict(H=256, I=128, B=4, T=16), dict(H=132, I=70, B=2, T=9)])
def test_backward_random_fp32(env, shape):
    """Random fp32 weights; the seed is the first one (from a fixed list)
    whose pre-activations all stay 1e-4 away from 0 in the oracle."""
    o = env[2]
    for seed in range(600, 640):
        p = synth.make_problem(seed=seed, wdtype="f32", h0_std=0.5, **shape)
        if _min_abs_preact(o, p) > 1e-4:
            break
    else:
        pytest.fail("no seed with pre-activations away from 0")
    dy = np.random.default_rng(seed).normal(size=(p.T, p.B, p.H))
    y, g = run(env, p, dy.astype(np.float32))
    ref = o.backward(p, dy.astype(np.float32))
    for k in ("delta", "dx", "dh0", "dWx", "dWh", "db"):
        assert rel_err(g[k], ref[k]) <= 1e-4, (k, rel_err(g[k], ref[k]))


def check_by_properties(env, p, dy, y, g, n_samples=300):
    """Teacher-forced reverse recurrence on sampled (t, b, r), and every
    gradient as its batched product of the GPU's own deltas."""
    o = env[2]
    Wh = p.Wh.astype(np.float64)
    d = g["delta"]
    rng = np.random.default_rng(7)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, n_samples), rng.integers(0, p.B, n_samples),
        rng.integers(0, p.H, n_samples))]
    samples += [(p.T - 1, 0, 0), (0, p.B - 1, p.H - 1)]
    want = o.delta_cells(Wh, samples, lambda t, b: dy[t, b], lambda t, b: y[t, b],
                         lambda t, b: None if t == p.T - 1 else d[t + 1, b])
    got = np.array([d[t, b, r] for t, b, r in samples])
    assert np.abs(got - want).max() <= 1e-4 * max(float(np.abs(d).max()), 1e-30)
    h0 = np.zeros((p.B, p.H)) if p.h0 is None else p.h0.astype(np.float64)
    prev = np.concatenate([h0[None], y[:-1]], axis=0)
    x = p.x.astype(np.float64)
    Wx = p.Wx.astype(np.float64)
    refs = {"db": d.sum(axis=(0, 1)),
            "dWh": np.einsum("tbr,tbc->rc", d, prev),
            "dWx": np.einsum("tbr,tbc->rc", d, x),
            "dx": np.einsum("tbr,rc->tbc", d, Wx),
            "dh0": d[0] @ Wh}
    for k, ref in refs.items():
        assert rel_err(g[k], ref) <= product_tol(p, k), (k, rel_err(g[k], ref))


# bf16 keeps 8 significant bits: each operand of a tensor-core gradient
# product is rounded by at most 2^-9 of itself, so each product term by at
# most ~2^-8, and a sum of such terms (fp32 accumulation) stays within 2^-8
# of the sum of the terms' magnitudes.  Relative to the largest gradient
# entry that is a few 2^-8 wherever the entries are of similar size; the
# bound used below is 2^-6 (4 x 2^-8).
BF16_PRODUCT_TOL = 2.0 ** -6


def product_tol(p, k):
    """fp16-weight layers form dWh (dense, or the stored values of sparse
    weights), dWx and dx on the tensor cores from bf16-rounded operands (fp32
    accumulation): BF16_PRODUCT_TOL of the scale; everything else is fp32
    arithmetic: 1e-4."""
    return BF16_PRODUCT_TOL if p.wdtype == "f16" and k in ("dWh", "dWx", "dx") else 1e-4


@pytest.mark.parametrize("spec", [dict(H=1152, B=4, T=32, wdtype="f16", h0_std=0.1),
                                  dict(H=260, I=96, B=7, T=11, wdtype="f16"),
                                  dict(H=4, I=4, B=2, T=3, wdtype="f32", h0_std=1.0),
                                  dict(H=640, B=32, T=3, wdtype="f16")])
def test_backward_properties(env, spec):
    p = synth.make_problem(seed=700, **spec)
    dy = np.random.default_rng(701).normal(size=(p.T, p.B, p.H)).astype(np.float32)
    y, g = run(env, p, dy)
    check_by_properties(env, p, dy.astype(np.float64), y, g)


def test_backward_full_size(env):
    """The dense fp16 H = 1152, B = 4 layer over the full 256 steps."""
    p = synth.named_problem("dense_f16_h1152_b4_t256")
    dy = np.random.default_rng(702).normal(size=(p.T, p.B, p.H)).astype(np.float32)
    y, g = run(env, p, dy)
    check_by_properties(env, p, dy.astype(np.float64), y, g, n_samples=400)


def test_backward_errors_and_edges(env):
    torch, prnn, _ = env
    p = synth.make_problem(H=64, B=2, T=3, wdtype="f16", seed=703)
    lay = prnn.prnn_create(64, 64, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    x = torch.from_numpy(p.x).cuda()
    y = torch.zeros(3, 2, 64, device="cuda")
    dy = torch.ones(3, 2, 64, device="cuda")
    db = torch.full((64,), 7.0, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_backward(lay, 3, 2, x, None, y, dy, db=db)
    assert e.value.status == prnn.PRNN_ERR_NOT_READY
    prnn.prnn_set_weights_dense(lay, torch.from_numpy(p.Wx).cuda(), torch.from_numpy(p.Wh).cuda(),
                                torch.from_numpy(p.b).cuda())
    prnn.prnn_backward(lay, 0, 2, x, None, y, dy, db=db)      # no steps: zero gradients
    torch.cuda.synchronize()
    assert torch.count_nonzero(db).item() == 0
    with pytest.raises(prnn.PrnnError) as e:                  # output overlaps an input
        prnn.prnn_backward(lay, 3, 2, x, None, y, dy, dx=x)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    big = torch.zeros(64 * 64 + 4, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:                  # misaligned output
        prnn.prnn_backward(lay, 3, 2, x, None, y, dy, dWh=big[1:].data_ptr())
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    prnn.prnn_destroy(lay)
    ps = prnn.prnn_create(64, 64, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PER_STEP)
    prnn.prnn_set_weights_dense(ps, torch.from_numpy(p.Wx).cuda(), torch.from_numpy(p.Wh).cuda(),
                                torch.from_numpy(p.b).cuda())
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_backward(ps, 3, 2, x, None, y, dy, db=db)
    assert e.value.status == prnn.PRNN_ERR_UNSUPPORTED
    prnn.prnn_destroy(ps)


def test_backward_dropped_publish_times_out(env):
    torch, prnn, o = env
    p = synth.make_problem(H=512, B=4, T=6, wdtype="f16", seed=704)
    lay = prnn.Layer.from_problem(p)
    x = torch.from_numpy(p.x).cuda()
    y = lay.forward(x)
    lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 3)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    lay.backward(x, y, torch.ones_like(y))
    assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    lay.close()


# --- sparse weights -------------------------------------------------------------
def dense_of(p):
    Wh = np.zeros((p.H, p.H))
    if getattr(p, "row_ptr", None) is not None:
        rows = np.repeat(np.arange(p.H), np.diff(p.row_ptr))
        Wh[rows, p.cols.astype(np.int64)] = p.vals.astype(np.float64)
    else:
        rows = np.repeat(np.arange(p.H), p.k)
        Wh[rows, p.cols.astype(np.int64).ravel()] = p.vals.astype(np.float64).ravel()
    return Wh


def dyadic_sparse_problem(seed, H, I, B, T, k, csr=False):
    """Row-balanced (or, with csr, rows of 0..2k entries) Wh of +-0.5 values;
    columns deliberately unsorted; every fp32 sum on the GPU exact."""
    rng = np.random.default_rng(seed)
    q = lambda *s: rng.integers(-8, 9, size=s).astype(np.float64) / 8
    if csr:
        lens = rng.integers(0, 2 * k + 1, size=H)
        lens[0] = 0
        row_ptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        cols = np.concatenate([rng.choice(H, n, replace=False) for n in lens]).astype(np.uint16)
        vals = rng.choice([-0.5, 0.5], size=int(lens.sum())).astype(np.float16)
    else:
        row_ptr = None
        cols = np.stack([rng.choice(H, k, replace=False) for _ in range(H)]).astype(np.uint16)
        vals = rng.choice([-0.5, 0.5], size=(H, k)).astype(np.float16)
    p = synth.Problem(name="dyadic_sparse", T=T, B=B, H=H, I=I, wdtype="f16",
                      x=q(T, B, I).astype(np.float32), Wx=(q(H, I) / 4).astype(np.float16),
                      b=q(H).astype(np.float32), h0=q(B, H).astype(np.float32), vals=vals,
                      cols=cols, row_ptr=row_ptr)
    return p, q(T, B, H)


@pytest.mark.parametrize("csr,staged", [(False, 0), (True, 0), (False, 1), (True, 1)])
@pytest.mark.parametrize("shape", [dict(H=64, I=32, B=3, T=6, k=3), dict(H=512, I=96, B=4, T=5, k=3)])
def test_sparse_backward_exact_problems(env, csr, staged, shape):
    """staged = 1: the forward and the reverse recurrence stage h / delta in
    each CTA's bank-balancing order (H = 512; H = 64 keeps column order)."""
    p, dy = dyadic_sparse_problem(800 + shape["H"], csr=csr, **shape)
    o = env[2]
    y, g = run(env, p, dy.astype(np.float32), {env[1].PRNN_OPT_PROJECTION: 1},
               pre_options={env[1].PRNN_OPT_STAGED_ORDER: staged})
    assert np.array_equal(y, o.forward(p)), "forward not exact: masks could differ"
    ref = o.backward(p, dy)
    assert rel_err(g["dWh"], ref["dvals"].ravel()) <= 1e-6
    for k in ("delta", "dx", "dh0", "dWx", "db"):
        assert rel_err(g[k], ref[k]) <= 1e-6, (k, rel_err(g[k], ref[k]))


def check_sparse_by_properties(env, p, dy, y, g, n_samples=300):
    o = env[2]
    Wh = dense_of(p)
    d = g["delta"]
    rng = np.random.default_rng(8)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, n_samples), rng.integers(0, p.B, n_samples),
        rng.integers(0, p.H, n_samples))]
    want = o.delta_cells(Wh, samples, lambda t, b: dy[t, b], lambda t, b: y[t, b],
                         lambda t, b: None if t == p.T - 1 else d[t + 1, b])
    got = np.array([d[t, b, r] for t, b, r in samples])
    assert np.abs(got - want).max() <= 1e-4 * max(float(np.abs(d).max()), 1e-30)
    h0 = np.zeros((p.B, p.H)) if p.h0 is None else p.h0.astype(np.float64)
    prev = np.concatenate([h0[None], y[:-1]], axis=0)
    dense_grad = np.einsum("tbr,tbc->rc", d, prev)
    if getattr(p, "row_ptr", None) is not None:
        rows = np.repeat(np.arange(p.H), np.diff(p.row_ptr))
        dvals = dense_grad[rows, p.cols.astype(np.int64)]
    else:
        dvals = dense_grad[np.repeat(np.arange(p.H), p.k), p.cols.astype(np.int64).ravel()]
    assert rel_err(g["dWh"], dvals) <= product_tol(p, "dWh")
    refs = {"db": d.sum(axis=(0, 1)), "dWx": np.einsum("tbr,tbc->rc", d, p.x.astype(np.float64)),
            "dx": np.einsum("tbr,rc->tbc", d, p.Wx.astype(np.float64)), "dh0": d[0] @ Wh}
    for k, ref in refs.items():
        assert rel_err(g[k], ref) <= product_tol(p, k), (k, rel_err(g[k], ref))


@pytest.mark.parametrize("name,T,staged", [("sparse_f16_h1792_d10_b4_t256", 32, 0),
                                           ("sparse_f16_h1792_d10_b4_t256", None, 0),
                                           ("sparse_f16_h5760_d1_b4_t256", 16, 0),
                                           ("sparse_f16_h1792_d10_b4_t256", 32, 1),
                                           ("sparse_f16_h5760_d5_b4_t256", 8, 1)])
def test_sparse_backward_properties(env, name, T, staged):
    p = synth.named_problem(name, T=T)
    dy = np.random.default_rng(705).normal(size=(p.T, p.B, p.H)).astype(np.float32)
    y, g = run(env, p, dy, pre_options={env[1].PRNN_OPT_STAGED_ORDER: staged})
    check_sparse_by_properties(env, p, dy.astype(np.float64), y, g)


def test_csr_backward_properties(env):
    p, _ = synth.make_pruned_pair(H=1792, B=4, T=24, density=0.10, seed=706)
    dy = np.random.default_rng(707).normal(size=(p.T, p.B, p.H)).astype(np.float32)
    y, g = run(env, p, dy)
    assert g["dWh"].shape == (p.nnz,)
    check_sparse_by_properties(env, p, dy.astype(np.float64), y, g)


@pytest.mark.parametrize("spec", [dict(H=1152, B=4, T=32, wdtype="f16"),
                                  dict(H=1792, B=4, T=16, k=179)])
def test_tensor_core_gradients_match_cuda_core(env, spec):
    """For the same forward output, the bf16 tensor-core products agree with
    the fp32 CUDA-core ones within the bf16 rounding of their operands, and
    delta, db and dh0 (fp32 on both paths) are bit-identical."""
    torch, prnn, _ = env
    p = synth.make_problem(seed=708, **spec)
    dy = torch.from_numpy(np.random.default_rng(709).normal(
        size=(p.T, p.B, p.H)).astype(np.float32)).cuda()
    lay = prnn.Layer.from_problem(p)
    try:
        x = torch.from_numpy(p.x).cuda()
        y = lay.forward(x)
        g_tc = {k: v.cpu().numpy().astype(np.float64) for k, v in lay.backward(x, y, dy).items()}
        lay.set_option(prnn.PRNN_OPT_PROJECTION, 1)
        g_cc = {k: v.cpu().numpy().astype(np.float64) for k, v in lay.backward(x, y, dy).items()}
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    for k in ("dWx", "dx", "dWh"):
        assert rel_err(g_tc[k], g_cc[k]) <= 1e-2, (k, rel_err(g_tc[k], g_cc[k]))
    for k in ("delta", "db", "dh0"):
        assert np.array_equal(g_tc[k], g_cc[k]), k


@pytest.mark.parametrize("kind", ["dense", "sparse", "csr"])
def test_ksplit_backward_exact_problems(env, kind):
    """At a wide batch the forward and the backward's reverse recurrence run
    on the tensor-core K-split kernel (Wh, then Wh^T; a sparse or CSR layer's
    densified matrix when forced on). On dyadic problems every h and delta
    splits exactly into fp16 hi + lo and every fp32 sum is exact, so the
    forward equals the oracle's bit for bit and delta, db, dh0 match the
    oracle's gradients within 1e-6 (the bf16 products within their bound)."""
    torch, prnn, o = env
    shape = dict(H=1152, I=1152, B=16, T=6)
    if kind == "dense":
        p, dy = dyadic_problem(960, wdtype="f16", **shape)
        opts = {}
    else:
        p, dy = dyadic_sparse_problem(961, k=3, csr=kind == "csr", **shape)
        opts = {prnn.PRNN_OPT_SPARSE_KSPLIT: 2}
    lay = prnn.Layer(p.H, p.I, p.B, p.wdtype, "persistent")
    try:
        for k, v in opts.items():
            lay.set_option(k, v)
        lay.set_problem_weights(p)
        assert lay.info()["dense_ksplit"] == 8  # H=1152: clusters of 8
    finally:
        lay.close()
    y, g = run(env, p, dy.astype(np.float32), options=opts or None, pre_options=opts or None)
    assert np.array_equal(y, o.forward(p)), "forward not exact: masks could differ"
    ref = o.backward(p, dy)
    for k in ("delta", "db", "dh0"):
        assert rel_err(g[k], ref[k]) <= 1e-6, (k, rel_err(g[k], ref[k]))
    for k in ("dWx", "dx", "dWh"):
        sparse = kind != "dense"
        want = ref["dvals"].ravel() if (sparse and k == "dWh") else ref[k]
        got = g[k].ravel() if (sparse and k == "dWh") else g[k]
        assert rel_err(got, want) <= BF16_PRODUCT_TOL, (k, rel_err(got, want))
    # the same gradients with the K-split kernel off
    off = {prnn.PRNN_OPT_DENSE_KSPLIT: 0, prnn.PRNN_OPT_SPARSE_KSPLIT: 0}
    _, g_off = run(env, p, dy.astype(np.float32), options=off, pre_options=off)
    assert np.array_equal(g["delta"], g_off["delta"])
