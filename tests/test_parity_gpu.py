"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Rule for every comparison, over the whole sequence:
    max |y_gpu - y_oracle| <= tol * max |y_oracle|
with tol = 1e-4 for fp32 weights and 2e-2 for fp16 weights (fp32 accumulation).
"""
import numpy as np
import pytest

import oracle
from persistent_rnn_recurrence_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2}


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    from persistent_rnn_recurrence_gb300 import prnn
    return torch, prnn, oracle.default()


def run_gpu(env, p, algo="persistent", T=None, max_batch=None, options=None, pre_options=None):
    """pre_options are set before the weights (options that act at set_weights)."""
    torch, prnn, _ = env
    if pre_options:
        lay = prnn.Layer(p.H, p.I, max_batch or max(1, p.B), p.wdtype, algo)
        for k, v in pre_options.items():
            lay.set_option(k, v)
        lay.set_problem_weights(p)
    else:
        lay = prnn.Layer.from_problem(p, algo=algo, max_batch=max_batch)
    try:
        for k, v in (options or {}).items():
            lay.set_option(k, v)
        x = torch.from_numpy(p.x if T is None else p.x[:T]).cuda()
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        st = lay.status()
        assert st == prnn.PRNN_OK, prnn.prnn_status_string(st)
        return y.cpu().numpy(), lay.info()
    finally:
        lay.close()


def check(y, ref, wdtype, what=""):
    scale = float(np.abs(ref).max())
    err = float(np.abs(y.astype(np.float64) - ref).max())
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    assert err <= TOL[wdtype] * scale, f"{what}: max err {err:.3e} vs {TOL[wdtype] * scale:.3e}"
    return err / max(scale, 1e-30)


# --- full-sequence parity: small and full configurations ----------------------
FULL = ["dense_f32_h256_b4_t32", "dense_f16_h1152_b4_t256", "sparse_f16_h1792_d10_b4_t256"]


@pytest.mark.parametrize("algo", ["persistent", "per_step"])
@pytest.mark.parametrize("name", FULL)
def test_named_full_sequence(env, name, algo):
    p = synth.named_problem(name)
    y, _ = run_gpu(env, p, algo)
    ref = env[2].forward(p)
    check(y, ref, p.wdtype, f"{name}/{algo}")


@pytest.mark.parametrize("algo", ["persistent", "per_step"])
@pytest.mark.parametrize("name", ["sparse_f16_h5760_d1_b4_t256", "sparse_f16_h5760_d5_b4_t256"])
def test_large_sparse_short_sequence(env, name, algo):
    p = synth.named_problem(name, T=8)
    y, _ = run_gpu(env, p, algo)
    check(y, env[2].forward(p), p.wdtype, f"{name}/{algo}")


@pytest.mark.parametrize("name", ["sparse_f16_h5760_d1_b4_t256", "sparse_f16_h5760_d5_b4_t256",
                                  "sparse_f16_h1792_d10_b4_t256"])
def test_full_size_teacher_forced_samples(env, name):
    """Full T = 256 in the benchmarked launch configuration: every sampled
    output must equal one oracle step applied to the GPU's own previous
    state, ReLU(b + Wx x_t + Wh y_gpu[t-1]) (a property that holds at any
    size), plus no sentinel or non-finite value anywhere."""
    p = synth.named_problem(name)
    y, _ = run_gpu(env, p)
    assert np.isfinite(y).all()
    rng = np.random.default_rng(5)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, 300), rng.integers(0, p.B, 300), rng.integers(0, p.H, 300))]
    samples += [(p.T - 1, p.B - 1, p.H - 1), (0, 0, 0)]
    h0 = np.zeros((p.B, p.H)) if p.h0 is None else p.h0
    got = np.array([y[t, b, r] for t, b, r in samples], dtype=np.float64)
    want = env[2].cells(p, samples, lambda t, b: p.x[t, b],
                        lambda t, b: h0[b] if t == 0 else y[t - 1, b])
    scale = float(np.abs(y).max())
    assert np.abs(got - want).max() <= TOL[p.wdtype] * scale


# --- ragged shapes and edge cases ----------------------------------------------
RAGGED = [
    dict(H=300, I=200, B=3, T=5, wdtype="f16", h0_std=0.3),
    dict(H=300, I=200, B=3, T=5, wdtype="f32", h0_std=0.3),
    dict(H=300, I=200, B=3, T=5, k=17),
    dict(H=260, I=96, B=1, T=7, k=3),
    dict(H=132, I=40, B=5, T=6, wdtype="f16"),            # two batch groups (dense)
    dict(H=132, I=40, B=9, T=4, k=12, h0_std=0.5),       # batch group of 16 (sparse)
    dict(H=640, I=640, B=32, T=3, k=64),                 # largest batch
    dict(H=640, I=640, B=32, T=3, wdtype="f16"),
    dict(H=4, I=4, B=2, T=3, wdtype="f32", h0_std=1.0),  # fewer rows than SMs
    dict(H=1024, I=64, B=4, T=1, k=1024 // 4, h0_std=1.0),  # T = 1
]


@pytest.mark.parametrize("algo", ["persistent", "per_step"])
@pytest.mark.parametrize("i", range(len(RAGGED)))
def test_ragged_shapes(env, i, algo):
    spec = dict(RAGGED[i])
    p = synth.make_problem(seed=100 + i, **spec)
    y, info = run_gpu(env, p, algo)
    check(y, env[2].forward(p), p.wdtype, f"ragged{i}/{algo}")


def test_wh_zero_gives_projection(env):
    """Wh = 0: y_t = ReLU(Wx x_t + b); exercises the projection alone."""
    p = synth.make_problem(H=384, I=320, B=4, T=6, wdtype="f16", seed=31, h0_std=1.0)
    p.Wh[:] = 0
    y, _ = run_gpu(env, p)
    ref = env[2].forward(p)
    check(y, ref, "f16", "wh0")
    # stronger than the rule: only the fp16 rounding of x separates them
    assert np.abs(y - ref).max() <= 5e-3 * np.abs(ref).max()


@pytest.mark.parametrize("spec", [dict(H=1792, B=4, T=64, k=179),
                                  dict(H=1152, I=320, B=32, T=79, k=115),
                                  dict(H=300, I=200, B=3, T=5, wdtype="f16"),
                                  dict(H=132, I=40, B=5, T=6, k=12)])
def test_tensor_core_projection_matches_cuda_core(env, spec):
    """The tcgen05 projection (x rounded to fp16, fp32 accumulation) and the
    fp32 CUDA-core projection agree within the fp16 rounding of x, and both
    paths stay within the oracle rule. The second shape (M = T*B = 2528 rows,
    a ragged last row tile) has more output tiles than a 152-SM GPU has SMs,
    so its GEMM runs with the 3-stage ring, two CTAs per SM."""
    _, prnn, o = env
    p = synth.make_problem(seed=33, **spec)
    y_tc, info = run_gpu(env, p)
    assert info["projection_tensor_cores"] == 1
    y_cc, info2 = run_gpu(env, p, options={prnn.PRNN_OPT_PROJECTION: 1})
    assert info2["projection_tensor_cores"] == 0
    ref = o.forward(p)
    check(y_tc, ref, "f16", "tc")
    check(y_cc, ref, "f16", "cuda cores")
    assert np.abs(y_tc - y_cc).max() <= 5e-3 * np.abs(ref).max()


def test_tensor_core_projection_ragged_rows(env):
    """H % 4 != 0 (the per-step path; the persistent kernels need H % 4 == 0):
    P's rows are not 16-byte multiples, so the tcgen05 projection stores its
    tiles thread by thread instead of by TMA, and still agrees with the
    CUDA-core projection and the oracle."""
    _, prnn, o = env
    p = synth.make_problem(H=301, I=77, B=3, T=5, wdtype="f16", seed=34, h0_std=0.3)
    y_tc, info = run_gpu(env, p, algo="per_step")
    assert info["projection_tensor_cores"] == 1
    y_cc, _ = run_gpu(env, p, algo="per_step", options={prnn.PRNN_OPT_PROJECTION: 1})
    ref = o.forward(p)
    check(y_tc, ref, "f16", "tc ragged")
    check(y_cc, ref, "f16", "cuda cores ragged")
    assert np.abs(y_tc - y_cc).max() <= 5e-3 * np.abs(ref).max()


def test_h0_none_equals_zeros(env):
    torch, prnn, _ = env
    p = synth.make_problem(H=256, B=2, T=4, k=20, seed=32)
    lay = prnn.Layer.from_problem(p)
    x = torch.from_numpy(p.x).cuda()
    y1 = lay.forward(x, None)
    y2 = lay.forward(x, torch.zeros(p.B, p.H, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    lay.close()


# --- exact properties of the CUDA path -----------------------------------------
@pytest.mark.parametrize("spec", [dict(H=1152, B=4, T=16, wdtype="f16"),
                                  dict(H=1792, B=4, T=16, k=179)])
def test_determinism_chaining_batch_independence(env, spec):
    torch, prnn, _ = env
    p = synth.make_problem(seed=41, h0_std=0.1, **spec)
    lay = prnn.Layer.from_problem(p)
    x = torch.from_numpy(p.x).cuda()
    h0 = torch.from_numpy(p.h0).cuda()
    y = lay.forward(x, h0)
    y_again = lay.forward(x, h0)
    # chaining: T1 steps then T2 steps from h0 = y[T1-1]
    ya = lay.forward(x[:7].contiguous(), h0)
    yb = lay.forward(x[7:].contiguous(), ya[-1].contiguous())
    # batch independence: each batch column alone
    ys = [lay.forward(x[:, b:b + 1].contiguous(), h0[b:b + 1].contiguous()) for b in range(p.B)]
    torch.cuda.synchronize()
    assert lay.status() == prnn.PRNN_OK
    assert torch.equal(y, y_again)
    assert torch.equal(torch.cat([ya, yb]), y)
    for b in range(p.B):
        assert torch.equal(ys[b][:, 0], y[:, b])
    lay.close()


@pytest.mark.parametrize("spec", [dict(H=1152, B=4, T=12, wdtype="f16"),
                                  dict(H=1792, B=4, T=12, k=179)])
def test_grid_barrier_mode_matches_flag_mode(env, spec):
    _, prnn, o = env
    p = synth.make_problem(seed=43, **spec)
    y0, _ = run_gpu(env, p)
    y1, _ = run_gpu(env, p, options={prnn.PRNN_OPT_SYNC_MODE: 1})
    assert np.array_equal(y0, y1)
    check(y1, o.forward(p), "f16", "gridbar")


@pytest.mark.parametrize("wide,bank,barrier", [(0, 0, 1), (1, 0, 1), (1, 1, 1), (0, 1, 0)])
def test_ablation_variants_match_oracle(env, wide, bank, barrier):
    """The ablation switches (32-bit staging loads, plain entry placement,
    grid barrier) change speed only: results stay within the rule."""
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=4, T=10, k=115, seed=44)
    lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
    lay.set_option(prnn.PRNN_OPT_BANK_AWARE, bank)
    lay.set_problem_weights(p)
    lay.set_option(prnn.PRNN_OPT_WIDE_LOADS, wide)
    lay.set_option(prnn.PRNN_OPT_SYNC_MODE, barrier)
    y = lay.forward(torch.from_numpy(p.x).cuda())
    assert lay.status() == prnn.PRNN_OK
    lay.close()
    check(y.cpu().numpy(), o.forward(p), "f16", f"ablation {wide}{bank}{barrier}")


# --- API behaviour ---------------------------------------------------------------
def test_plan_report(env):
    _, prnn, _ = env
    p = synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=2)
    lay = prnn.Layer.from_problem(p)
    info = lay.info()
    lay.close()
    assert info["sparse"] == 1 and info["k"] == 179 and info["nnz"] == 1792 * 179
    assert info["k_padded"] % (4 * info["threads_per_row"]) == 0
    assert info["n_cta"] * info["rows_per_cta"] >= 1792
    assert info["n_cta"] <= info["sm_count"]
    assert info["onchip_weight_bytes"] == (info["n_cta"] * info["rows_per_cta"]
                                           * info["k_padded"] * 4)


def test_errors(env):
    torch, prnn, _ = env
    p = synth.make_problem(H=64, B=2, T=3, k=8, seed=50)
    lay = prnn.prnn_create(64, 64, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    x = torch.from_numpy(p.x).cuda()
    y = torch.empty(3, 2, 64, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_forward(lay, 3, 2, x, None, y)
    assert e.value.status == prnn.PRNN_ERR_NOT_READY
    Wx = torch.from_numpy(p.Wx).cuda()
    b = torch.from_numpy(p.b).cuda()
    vals = torch.from_numpy(p.vals.view(np.int16)).cuda()
    bad = p.cols.copy()
    bad[5, 1] = bad[5, 0]                                     # duplicate column
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_set_weights_sparse(lay, Wx, 8, vals, torch.from_numpy(bad.view(np.int16)).cuda(), b)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    bad = p.cols.copy()
    bad[0, 0] = 64                                            # out of range
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_set_weights_sparse(lay, Wx, 8, vals, torch.from_numpy(bad.view(np.int16)).cuda(), b)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    prnn.prnn_set_weights_sparse(lay, Wx, 8, vals, torch.from_numpy(p.cols.view(np.int16)).cuda(), b)
    for B_, what in ((3, "B > max_batch"),):
        with pytest.raises(prnn.PrnnError) as e:
            prnn.prnn_forward(lay, 3, B_, x, None, y)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG, what
    ybig = torch.empty(3 * 2 * 64 + 4, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:                   # misaligned y
        prnn.prnn_forward(lay, 3, 2, x, None, ybig[1:].data_ptr())
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    with pytest.raises(prnn.PrnnError) as e:                   # y overlaps x
        prnn.prnn_forward(lay, 3, 2, x, None, x)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    prnn.prnn_forward(lay, 0, 2, x, None, y)                   # T = 0: no-op
    prnn.prnn_forward(lay, 3, 0, x, None, y)                   # B = 0: no-op
    assert prnn.prnn_get_status(lay) == prnn.PRNN_OK
    prnn.prnn_destroy(lay)
    # uint16 column indices: a sparse layer needs H <= 65535
    wide = prnn.prnn_create(65536, 64, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_set_weights_sparse(wide, Wx, 8, vals, torch.from_numpy(p.cols.view(np.int16)).cuda(), b)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    prnn.prnn_destroy(wide)
    # a dense layer too large for the chip is refused, not silently degraded
    big = prnn.prnn_create(8192, 64, 4, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    Wh = torch.zeros(8192, 8192, dtype=torch.float16, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_set_weights_dense(big, torch.zeros(8192, 64, dtype=torch.float16, device="cuda"),
                                    Wh, torch.zeros(8192, device="cuda"))
    assert e.value.status == prnn.PRNN_ERR_UNSUPPORTED
    prnn.prnn_destroy(big)


def test_host_weight_pointers(env):
    """set_weights accepts host memory too (the library copies)."""
    torch, prnn, o = env
    p = synth.make_problem(H=256, B=2, T=5, k=25, seed=51)
    lay = prnn.prnn_create(256, 256, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    prnn.prnn_set_weights_sparse(lay, p.Wx.ctypes.data, p.k, p.vals.ctypes.data,
                                 p.cols.ctypes.data, p.b.ctypes.data)
    x = torch.from_numpy(p.x).cuda()
    y = torch.empty(5, 2, 256, device="cuda")
    prnn.prnn_forward(lay, 5, 2, x, None, y)
    assert prnn.prnn_get_status(lay) == prnn.PRNN_OK
    prnn.prnn_destroy(lay)
    check(y.cpu().numpy(), o.forward(p), "f16", "host pointers")


# --- unbalanced compressed rows (global magnitude pruning) ---------------------------
@pytest.mark.parametrize("algo", ["persistent", "per_step"])
@pytest.mark.parametrize("spec", [dict(H=300, B=3, T=6, density=0.05, row_sigma=1.0),
                                  dict(H=40, B=2, T=5, density=0.1, row_sigma=1.0),
                                  dict(H=2304, B=4, T=12, density=0.25, row_sigma=0.25)])
def test_csr_unbalanced_matches_oracle(env, spec, algo):
    """Rows of unequal length, empty rows included: the library pads each row
    to the longest one; the result is that of the compressed-row definition."""
    unb, bal = synth.make_pruned_pair(seed=70, **spec)
    assert (np.diff(unb.row_ptr) != unb.k).any()
    for p in (unb, bal):
        y, info = run_gpu(env, p, algo)
        assert info["k"] == p.k
        check(y, env[2].forward(p), "f16", f"{p.name}/{algo}")


def test_csr_full_size_teacher_forced_samples(env):
    """The 25 %-dense H = 2304 globally pruned layer at T = 256 in the
    benchmarked configuration, checked by one oracle step per sampled output
    applied to the GPU's own previous state."""
    p, _ = synth.make_pruned_pair(H=2304, B=4, T=256, density=0.25, seed=71)
    y, _ = run_gpu(env, p)
    assert np.isfinite(y).all()
    rng = np.random.default_rng(6)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, 200), rng.integers(0, p.B, 200), rng.integers(0, p.H, 200))]
    samples.append((p.T - 1, p.B - 1, int(np.argmax(np.diff(p.row_ptr)))))
    got = np.array([y[t, b, r] for t, b, r in samples], dtype=np.float64)
    want = env[2].cells(p, samples, lambda t, b: p.x[t, b],
                        lambda t, b: np.zeros(p.H) if t == 0 else y[t - 1, b])
    assert np.abs(got - want).max() <= TOL["f16"] * float(np.abs(y).max())


def test_csr_errors(env):
    torch, prnn, _ = env
    p, _ = synth.make_pruned_pair(H=64, B=2, T=3, density=0.1, seed=72, row_sigma=1.0)
    lay = prnn.prnn_create(64, 64, 2, prnn.PRNN_F16, prnn.PRNN_ALGO_PERSISTENT)
    Wx = torch.from_numpy(p.Wx).cuda()
    b = torch.from_numpy(p.b).cuda()
    vals = torch.from_numpy(p.vals.view(np.int16)).cuda()
    nnz = p.nnz

    def put(rp, cols, n=nnz):
        return prnn.prnn_set_weights_csr(
            lay, Wx, n, torch.from_numpy(rp.astype(np.int32)).cuda(),
            torch.from_numpy(cols.view(np.int16)).cuda(), vals, b)

    bad_rp = p.row_ptr.copy()
    bad_rp[10], bad_rp[11] = bad_rp[11] + 1, bad_rp[10]       # decreasing offsets
    for rp, cols, n in ((bad_rp, p.cols, nnz), (p.row_ptr, p.cols, nnz - 1)):
        with pytest.raises(prnn.PrnnError) as e:
            put(rp, cols, n)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    lens = np.diff(p.row_ptr)
    r = int(np.argmax(lens >= 2))
    dup = p.cols.copy()
    dup[p.row_ptr[r] + 1] = dup[p.row_ptr[r]]                 # duplicate column in a row
    oob = p.cols.copy()
    oob[0] = 64                                               # column out of range
    for cols in (dup, oob):
        with pytest.raises(prnn.PrnnError) as e:
            put(p.row_ptr, cols)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    put(p.row_ptr, p.cols)
    assert prnn.prnn_get_info(lay)["k"] == int(lens.max())
    prnn.prnn_destroy(lay)


# --- bounded waits: a publish that never happens ends in a status, not a hang --------
@pytest.mark.parametrize("spec", [dict(H=512, B=4, T=6, k=40), dict(H=512, B=4, T=6, wdtype="f16")])
def test_dropped_publish_times_out_cleanly(env, spec):
    torch, prnn, o = env
    p = synth.make_problem(seed=60, **spec)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 3)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    x = torch.from_numpy(p.x).cuda()
    lay.forward(x)
    assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    with pytest.raises(prnn.PrnnError) as e:                   # sticky
        lay.forward(x)
    assert e.value.status == prnn.PRNN_ERR_TIMEOUT
    lay.close()
    # the context is still usable: a fresh handle computes correctly
    y, _ = run_gpu(env, p)
    check(y, o.forward(p), "f16", "after timeout")


def test_sync_floor_probe(env):
    torch, prnn, _ = env
    p = synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=2)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_TIMING, 1)
    y = torch.empty(64, 4, 1792, device="cuda")
    prnn.prnn_probe_sync_floor(lay.h, 64, 4, y)
    assert lay.status() == prnn.PRNN_OK
    _, ms = prnn.prnn_get_timing(lay.h)
    lay.close()
    t = torch.arange(1, 65, dtype=torch.float32, device="cuda").view(64, 1, 1)
    assert torch.equal(y, t.expand(64, 4, 1792))
    assert ms > 0


@pytest.mark.parametrize("spec", [dict(H=1792, B=4, T=24, k=179),
                                  dict(H=5760, B=4, T=10, k=57, h0_std=0.2),
                                  dict(H=1152, B=2, T=16, k=230),
                                  dict(H=640, B=3, T=9, k=96),
                                  dict(H=2304, B=16, T=8, k=230),
                                  dict(H=4096, B=4, T=6, k=409, h0_std=0.2)])
def test_register_weight_build_gives_the_same_bits(env, spec):
    """The register-weight build of the sparse kernel (384-thread launch
    bound, 24 entries per thread in registers) and the plan-matched staging
    depth (2 or 6 float4 loads in flight instead of 12) change where values
    wait, not what is summed in which order: every on/off combination gives
    the same bits, forward and backward, within the rule of the oracle."""
    torch, prnn, o = env
    p = synth.make_problem(seed=86, **spec)
    ys, deltas = [], []
    for regw, depth in ((1, 1), (0, 0), (1, 0), (0, 1)):
        lay = prnn.Layer.from_problem(p)
        try:
            lay.set_option(prnn.PRNN_OPT_SPARSE_KSPLIT, 0)  # the sparse kernel's builds
            lay.set_option(prnn.PRNN_OPT_SPARSE_REG_WEIGHTS, regw)
            lay.set_option(prnn.PRNN_OPT_SPARSE_STAGING_DEPTH, depth)
            info = lay.info()
            x = torch.from_numpy(p.x).cuda()
            h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
            y = lay.forward(x, h0)
            dy = torch.ones_like(y)
            g = lay.backward(x, y, dy, h0)
            torch.cuda.synchronize()
            assert lay.status() == prnn.PRNN_OK
        finally:
            lay.close()
        ys.append(y)
        deltas.append(g["delta"])
        fits = info["threads_per_cta"] <= 384 and info["k_padded"] // info["threads_per_row"] >= 24
        assert info["sparse_reg_weights"] == (1 if fits and regw else 0)
    for y, d in zip(ys[1:], deltas[1:]):
        assert torch.equal(ys[0], y) and torch.equal(deltas[0], d)
    check(ys[0].cpu().numpy(), o.forward(p), "f16", "register weights")
    lay = prnn.Layer.from_problem(p)
    try:
        for opt in (prnn.PRNN_OPT_SPARSE_REG_WEIGHTS, prnn.PRNN_OPT_SPARSE_STAGING_DEPTH):
            with pytest.raises(prnn.PrnnError) as e:
                lay.set_option(opt, 2)
            assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    finally:
        lay.close()


@pytest.mark.parametrize("spec", [dict(H=1792, B=4, T=12, k=179), dict(H=300, B=9, T=7, k=17)])
def test_phase_trace(env, spec):
    """The phase-trace build of the sparse kernel gives the same bits as the
    default build and writes one well-formed record per step and working CTA:
    its CTA index, an SM id below the SM count, its warp count, and per warp
    stamps in phase order; CTAs without batch columns write nothing."""
    torch, prnn, o = env
    p = synth.make_problem(seed=84, **spec)
    W = 17 * 16
    lay = prnn.Layer.from_problem(p)
    try:
        info = lay.info()
        n = info["n_cta"]
        x = torch.from_numpy(p.x).cuda()
        y0 = lay.forward(x)
        buf = torch.full((p.T * n * W,), -1, dtype=torch.int32, device="cuda")
        with pytest.raises(prnn.PrnnError) as e:                # too small for T steps
            prnn.prnn_set_trace_buffer(lay.h, buf, buf.numel() * 4 - 16)
            lay.forward(x)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
        with pytest.raises(prnn.PrnnError) as e:                # host memory
            prnn.prnn_set_trace_buffer(lay.h, buf.cpu().data_ptr(), buf.numel() * 4)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
        prnn.prnn_set_trace_buffer(lay.h, buf, buf.numel() * 4)
        y1 = lay.forward(x)
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
        prnn.prnn_set_trace_buffer(lay.h, None, 0)
        y2 = lay.forward(x)
        torch.cuda.synchronize()
    finally:
        lay.close()
    assert torch.equal(y0, y1) and torch.equal(y0, y2)
    check(y1.cpu().numpy(), o.forward(p), "f16", "traced")
    rec = buf.view(p.T, n, 17, 16).cpu().numpy().view(np.uint32).astype(np.int64)
    G = info["cta_groups"]
    bl = -(-p.B // G)
    active = np.array([(c // (n // G)) * bl < p.B for c in range(n)])
    assert active.any()
    assert (rec[:, ~active] == 0xffffffff).all()
    rec = rec[:, active]
    nw = info["threads_per_cta"] // 32
    assert (rec[:, :, 0, 1] == np.arange(n)[active][None, :]).all()
    assert (rec[:, :, 0, 0] < info["sm_count"]).all()
    assert (rec[:, :, 0, 2] == nw).all()
    assert (rec[:, :, 1 + nw:] == 0xffffffff).all()
    stamps = rec[:, :, 1:1 + nw, :8]
    gaps = np.diff(stamps, axis=3) & 0xffffffff
    assert (gaps < (1 << 28)).all()             # every phase ends after the one before it
    gbar = (rec[:, :, 1:1 + nw, 10] << 32) | rec[:, :, 1:1 + nw, 9]
    gpub = (rec[:, :, 1:1 + nw, 12] << 32) | rec[:, :, 1:1 + nw, 11]
    assert (gpub >= gbar).all() and (np.diff(gpub.max(axis=2), axis=0) > 0).all()
    # a dense layer outside the K-split kernel has no traced kernel
    q = synth.make_problem(H=256, B=2, T=3, wdtype="f16", seed=85)
    lay = prnn.Layer.from_problem(q)
    try:
        prnn.prnn_set_trace_buffer(lay.h, buf, buf.numel() * 4)
        with pytest.raises(prnn.PrnnError) as e:
            lay.forward(torch.from_numpy(q.x).cuda())
        assert e.value.status == prnn.PRNN_ERR_UNSUPPORTED
    finally:
        lay.close()


@pytest.mark.parametrize("spec", [dict(H=1152, B=4, T=20, wdtype="f16"),
                                  dict(H=1792, B=4, T=20, k=179)])
def test_poll_delay_changes_timing_not_results(env, spec):
    """The pause before each step's first poll only shifts when data is read:
    results are bit-identical for 0, the default and a long pause."""
    torch, prnn, o = env
    p = synth.make_problem(seed=80, **spec)
    ys = []
    for d in (None, 0, 2000):
        y, _ = run_gpu(env, p, options={} if d is None else {prnn.PRNN_OPT_POLL_DELAY_NS: d})
        ys.append(y)
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])
    check(ys[0], o.forward(p), p.wdtype, "poll delay")
    lay = prnn.Layer.from_problem(p)
    with pytest.raises(prnn.PrnnError) as e:
        lay.set_option(prnn.PRNN_OPT_POLL_DELAY_NS, -1)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    lay.close()


@pytest.mark.parametrize("spec", [dict(H=1792, B=4, T=24, k=179),
                                  dict(H=1152, B=9, T=10, k=115, h0_std=0.5),
                                  dict(H=256, B=32, T=6, k=40),
                                  dict(H=300, B=3, T=8, k=17)])
def test_staged_order_matches_column_order(env, spec):
    """Each CTA staging h_{t-1} in its own bank-balancing order changes where
    the gathers read, not what they read: both orders match the oracle, and
    ragged H (not a multiple of 128) keeps column order.  At these sizes the
    automatic choice (the default) is column order."""
    torch, prnn, o = env
    p = synth.make_problem(seed=81, **spec)
    ref = o.forward(p)
    y_on, info_on = run_gpu(env, p, pre_options={prnn.PRNN_OPT_STAGED_ORDER: 1})
    y_off, info_off = run_gpu(env, p, pre_options={prnn.PRNN_OPT_STAGED_ORDER: 0})
    _, info_auto = run_gpu(env, p)
    assert info_auto["sparse_staged_order"] == 0
    check(y_on, ref, "f16", "staged order")
    check(y_off, ref, "f16", "column order")
    assert info_on["sparse_staged_order"] == (1 if p.H % 128 == 0 else 0)
    assert info_off["sparse_staged_order"] == 0
    if p.H % 128 == 0:
        assert info_on["sparse_bank_cap"] <= info_off["sparse_bank_cap"]
    # the same through the narrow (32-bit) staging of the ablation
    y_nar, _ = run_gpu(env, p, options={prnn.PRNN_OPT_WIDE_LOADS: 0},
                       pre_options={prnn.PRNN_OPT_STAGED_ORDER: 1})
    check(y_nar, ref, "f16", "staged order, narrow staging")
    lay = prnn.Layer.from_problem(p)
    try:
        with pytest.raises(prnn.PrnnError) as e:
            lay.set_option(prnn.PRNN_OPT_STAGED_ORDER, 3)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    finally:
        lay.close()


def test_staged_order_automatic_choice(env):
    """By default each packing picks its staging order by the measured rule:
    the staged order for a wide batch of a 25 % layer, column order for the
    headline layer (B = 4); the chosen forwards match the oracle."""
    _, prnn, o = env
    p = synth.make_problem(H=2304, B=32, T=6, k=576, seed=82, h0_std=0.3)
    # the sparse kernel (by default this layer runs its densified matrix on
    # the K-split kernel)
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_SPARSE_KSPLIT: 0})
    assert info["sparse_staged_order"] == 1 and info["dense_ksplit"] == 0
    check(y, o.forward(p), "f16", "automatic staging order")
    q = synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=4)
    yq, info_q = run_gpu(env, q)
    assert info_q["sparse_staged_order"] == 0
    check(yq, o.forward(q), "f16", "automatic staging order, headline")
    # every named sparse layer (B = 4: one column a pass) keeps column order,
    # including H=5760 5 %, where the staged order packs tighter yet is slower
    for name in [n for n in synth.NAMED if n.startswith("sparse")]:
        lay = prnn.Layer.from_problem(synth.named_problem(name, T=1))
        try:
            assert lay.info()["sparse_staged_order"] == 0, name
        finally:
            lay.close()


@pytest.mark.parametrize("spec,algo,opts", [
    (dict(H=1792, B=4, T=40, k=179), "persistent", {}),
    (dict(H=1152, B=4, T=24, wdtype="f16", h0_std=0.3), "persistent", {}),
    (dict(H=256, I=100, B=5, T=9, wdtype="f32", h0_std=0.5), "persistent", {}),
    (dict(H=300, B=3, T=7, k=17), "per_step", {}),
    (dict(H=1152, B=16, T=8, wdtype="f16"), "persistent", {"PRNN_OPT_RECURRENT_TC": 2}),
    (dict(H=1152, B=24, T=10, wdtype="f16", h0_std=0.2), "persistent", {}),
    (dict(H=512, B=4, T=6, k=51), "persistent", {"PRNN_OPT_SYNC_MODE": 1})])
def test_forward_host_buffers(env, spec, algo, opts):
    """prnn_forward_host on pinned host buffers gives the bits prnn_forward
    gives on device copies (persistent kernels write y over the host link; the
    per-step path and the tcgen05 dense recurrence copy it back), and refuses
    pageable and device memory."""
    torch, prnn, o = env
    p = synth.make_problem(seed=83, **spec)
    pre = {getattr(prnn, k): v for k, v in opts.items() if k == "PRNN_OPT_RECURRENT_TC"}
    post = {getattr(prnn, k): v for k, v in opts.items() if k != "PRNN_OPT_RECURRENT_TC"}
    y_dev, _ = run_gpu(env, p, algo=algo, options=post, pre_options=pre or None)
    if pre:
        lay = prnn.Layer(p.H, p.I, max(1, p.B), p.wdtype, algo)
        for k, v in pre.items():
            lay.set_option(k, v)
        lay.set_problem_weights(p)
    else:
        lay = prnn.Layer.from_problem(p, algo=algo)
    try:
        for k, v in post.items():
            lay.set_option(k, v)
        xh = torch.from_numpy(p.x).pin_memory()
        h0h = None if p.h0 is None else torch.from_numpy(p.h0).pin_memory()
        yh = torch.full((p.T, p.B, p.H), -1.0).pin_memory()
        for _ in range(2):  # twice: the workspaces are reused
            prnn.prnn_forward_host(lay.h, p.T, p.B, xh, h0h, yh)
            torch.cuda.synchronize()
            assert lay.status() == prnn.PRNN_OK
            assert np.array_equal(yh.numpy(), y_dev)
        with pytest.raises(prnn.PrnnError) as e:           # pageable host memory
            prnn.prnn_forward_host(lay.h, p.T, p.B, torch.from_numpy(p.x.copy()), None, yh)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
        with pytest.raises(prnn.PrnnError) as e:           # device memory
            prnn.prnn_forward_host(lay.h, p.T, p.B, xh, None, yh.cuda())
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    finally:
        lay.close()
    check(y_dev, o.forward(p), p.wdtype, "host buffers")


# --- tensor-core dense recurrence (wide batches) --------------------------------------
@pytest.mark.parametrize("spec,force", [(dict(H=1152, B=16, T=64, wdtype="f16"), 0),
                                        (dict(H=2304, B=32, T=24, wdtype="f16", h0_std=0.2), 0),
                                        (dict(H=640, I=200, B=20, T=12, wdtype="f16"), 0),
                                        (dict(H=1152, B=4, T=32, wdtype="f16"), 2),
                                        (dict(H=128, B=9, T=7, wdtype="f16", h0_std=1.0), 2)])
def test_tensor_core_recurrence_matches_oracle(env, spec, force):
    torch, prnn, o = env
    p = synth.make_problem(seed=90, **spec)
    lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
    try:
        if force is not None:
            lay.set_option(prnn.PRNN_OPT_RECURRENT_TC, force)
        lay.set_problem_weights(p)
        assert lay.info()["recurrent_tensor_cores"] == 1
        x = torch.from_numpy(p.x).cuda()
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    check(y.cpu().numpy(), o.forward(p), "f16", f"tc {spec}")


def test_tensor_core_recurrence_off_and_fallback(env):
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=16, T=8, wdtype="f16", seed=91)
    y_tc, info = run_gpu(env, p, options=None)
    assert info["recurrent_tensor_cores"] == 0  # opt-in
    lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
    lay.set_option(prnn.PRNN_OPT_RECURRENT_TC, 2)
    lay.set_problem_weights(p)
    assert lay.info()["recurrent_tensor_cores"] == 1
    y_on = lay.forward(torch.from_numpy(p.x).cuda()).cpu().numpy()
    lay.close()
    ref = o.forward(p)
    check(y_tc, ref, "f16", "cuda cores")
    check(y_on, ref, "f16", "tensor cores")
    # H not a multiple of 64: CUDA-core kernel even when asked
    q = synth.make_problem(H=300, B=16, T=4, wdtype="f16", seed=92)
    y, info = run_gpu(env, q, pre_options={prnn.PRNN_OPT_RECURRENT_TC: 2})
    assert info["recurrent_tensor_cores"] == 0
    check(y, o.forward(q), "f16", "fallback")


def test_tensor_core_recurrence_full_size_teacher_forced(env):
    """H = 2304, B = 32, T = 256 (a sweep point): sampled outputs against one
    oracle step on the GPU's own previous state."""
    torch, prnn, o = env
    p = synth.make_problem(H=2304, B=32, T=256, wdtype="f16", seed=93)
    y, info = run_gpu(env, p, pre_options={prnn.PRNN_OPT_RECURRENT_TC: 2})
    assert info["recurrent_tensor_cores"] == 1 and np.isfinite(y).all()
    rng = np.random.default_rng(10)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, 200), rng.integers(0, p.B, 200), rng.integers(0, p.H, 200))]
    got = np.array([y[t, b, r] for t, b, r in samples], dtype=np.float64)
    want = o.cells(p, samples, lambda t, b: p.x[t, b],
                   lambda t, b: np.zeros(p.H) if t == 0 else y[t - 1, b])
    assert np.abs(got - want).max() <= TOL["f16"] * float(np.abs(y).max())


def test_tensor_core_recurrence_times_out_cleanly(env):
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=16, T=6, wdtype="f16", seed=94)
    lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
    lay.set_option(prnn.PRNN_OPT_RECURRENT_TC, 2)
    lay.set_problem_weights(p)
    assert lay.info()["recurrent_tensor_cores"] == 1
    lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 5)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    lay.forward(torch.from_numpy(p.x).cuda())
    assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    lay.close()
    y, _ = run_gpu(env, p)
    check(y, o.forward(p), "f16", "after timeout")


# --- dense fp16, wide batches: weights in registers, passes of 8 columns ------------
WIDE = [dict(H=2304, B=32, T=24, wdtype="f16", h0_std=0.2),  # 16 rows per CTA, 4 passes
        dict(H=1152, B=32, T=40, wdtype="f16"),              # 8 rows per CTA
        dict(H=1152, B=16, T=40, wdtype="f16"),              # 2 passes
        dict(H=1152, B=21, T=20, wdtype="f16", h0_std=0.5),  # passes of 8 + 8 + 5
        dict(H=640, I=200, B=24, T=16, wdtype="f16", h0_std=1.0),
        dict(H=256, B=17, T=30, wdtype="f16"),               # passes of 8 + 8 + 1
        dict(H=1792, B=20, T=20, wdtype="f16"),
        dict(H=1024, B=16, T=20, wdtype="f16"),
        dict(H=2048, B=16, T=12, wdtype="f16", h0_std=0.3),
        dict(H=128, I=64, B=32, T=50, wdtype="f16")]         # 4 weights per thread


@pytest.mark.parametrize("spec", WIDE)
def test_dense_wide_batch_matches_oracle(env, spec):
    """The wide-batch kernel (forced on for every B >= 16) and the B <= 4
    kernel both stay within the rule."""
    _, prnn, o = env
    p = synth.make_problem(seed=95, **spec)
    ref = o.forward(p)
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_WIDE: 2,
                                       prnn.PRNN_OPT_DENSE_KSPLIT: 0})
    assert info["dense_wide_batch"] == 1 and info["rows_per_cta"] in (8, 16)
    assert info["n_cta"] == p.H // info["rows_per_cta"] <= info["sm_count"]
    check(y, ref, "f16", f"wide {spec}")
    y_old, info_old = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_WIDE: 0,
                                               prnn.PRNN_OPT_DENSE_KSPLIT: 0})
    assert info_old["dense_wide_batch"] == 0 and info_old["dense_ksplit"] == 0
    check(y_old, ref, "f16", f"wide off {spec}")


def test_dense_wide_batch_exact_properties(env):
    """Determinism, chaining, and batch independence across the forwards that
    run the wide kernel (a column's arithmetic does not depend on its pass or
    neighbours); a forward of fewer than 16 columns runs the B <= 4 kernel
    and stays within the rule."""
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=32, T=16, wdtype="f16", seed=96, h0_std=0.1)
    lay = prnn.Layer.from_problem(p)
    try:
        lay.set_option(prnn.PRNN_OPT_DENSE_KSPLIT, 0)
        assert lay.info()["dense_wide_batch"] == 1  # by default: 4 passes, H >= 1024
        lay.set_option(prnn.PRNN_OPT_DENSE_WIDE, 2)  # and for the B = 16 forwards below
        info = lay.info()
        assert info["dense_wide_batch"] == 1 and info["cta_groups"] == 1
        assert info["n_cta"] == 144 and info["threads_per_cta"] == 192  # 2 x 96
        x = torch.from_numpy(p.x).cuda()
        h0 = torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        y_again = lay.forward(x, h0)
        ya = lay.forward(x[:7].contiguous(), h0)
        yb = lay.forward(x[7:].contiguous(), ya[-1].contiguous())
        y16a = lay.forward(x[:, :16].contiguous(), h0[:16].contiguous())
        y16b = lay.forward(x[:, 16:].contiguous(), h0[16:].contiguous())
        y20 = lay.forward(x[:, 5:25].contiguous(), h0[5:25].contiguous())
        y10 = lay.forward(x[:, :10].contiguous(), h0[:10].contiguous())  # B <= 4 kernel
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    assert torch.equal(y, y_again)
    assert torch.equal(torch.cat([ya, yb]), y)
    assert torch.equal(torch.cat([y16a, y16b], dim=1), y)
    assert torch.equal(y20, y[:, 5:25])
    ref = o.forward(p)
    check(y.cpu().numpy(), ref, "f16", "wide")
    check(y10.cpu().numpy(), ref[:, :10], "f16", "fallback at 10 columns")


def test_dense_wide_batch_full_size_teacher_forced(env):
    """H = 2304, B = 32, T = 256 (a sweep point): sampled outputs against one
    oracle step on the GPU's own previous state."""
    _, _, o = env
    _, prnn, _ = env
    p = synth.make_problem(H=2304, B=32, T=256, wdtype="f16", seed=97)
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_KSPLIT: 0})
    assert info["dense_wide_batch"] == 1 and np.isfinite(y).all()
    rng = np.random.default_rng(11)
    samples = [(int(t), int(b), int(r)) for t, b, r in zip(
        rng.integers(0, p.T, 300), rng.integers(0, p.B, 300), rng.integers(0, p.H, 300))]
    got = np.array([y[t, b, r] for t, b, r in samples], dtype=np.float64)
    want = o.cells(p, samples, lambda t, b: p.x[t, b],
                   lambda t, b: np.zeros(p.H) if t == 0 else y[t - 1, b])
    assert np.abs(got - want).max() <= TOL["f16"] * float(np.abs(y).max())


def test_dense_wide_batch_default_rule(env):
    """Option 1 (default) runs the wide kernel only where it measured faster;
    option 0 never; option 2 for every B >= 16."""
    _, prnn, _ = env
    cases = [(1152, 32, 1), (1152, 16, 0), (2304, 16, 1), (2304, 32, 1), (640, 32, 0),
             (1152, 8, 0)]
    for H, B, want in cases:
        lay = prnn.Layer(H, H, B, "f16", "persistent")
        try:
            p = synth.make_problem(H=H, B=B, T=1, wdtype="f16", seed=99)
            lay.set_problem_weights(p)
            lay.set_option(prnn.PRNN_OPT_DENSE_KSPLIT, 0)
            assert lay.info()["dense_wide_batch"] == want, (H, B)
            lay.set_option(prnn.PRNN_OPT_DENSE_WIDE, 0)
            assert lay.info()["dense_wide_batch"] == 0
            lay.set_option(prnn.PRNN_OPT_DENSE_WIDE, 2)
            assert lay.info()["dense_wide_batch"] == (1 if B >= 16 else 0)
            with pytest.raises(prnn.PrnnError):
                lay.set_option(prnn.PRNN_OPT_DENSE_WIDE, 3)
        finally:
            lay.close()


def test_dense_wide_batch_times_out_cleanly(env):
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=24, T=6, wdtype="f16", seed=98)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_DENSE_KSPLIT, 0)
    assert lay.info()["dense_wide_batch"] == 1
    lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 5)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    lay.forward(torch.from_numpy(p.x).cuda())
    assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    lay.close()
    y, _ = run_gpu(env, p)
    check(y, o.forward(p), "f16", "after timeout")


# --- the cluster exchange probe (a diagnostic of the step exchange) --------------------
def test_cluster_exchange_probe(env):
    """Every word pushed through distributed shared memory arrives with its
    value, at every cluster size; more clusters than the device can hold at
    once are refused."""
    _, prnn, _ = env
    for cs, ncl in ((2, 8), (4, 8), (8, 4), (16, 2), (16, 1)):
        ns, bad = prnn.prnn_probe_cluster_exchange(1792, cs, ncl, 200)
        assert bad == 0, (cs, ncl)
        assert 0.0 < ns < 1e5, (cs, ncl, ns)
    ns, bad = prnn.prnn_probe_cluster_exchange(5760, 16, 1, 50)
    assert bad == 0 and ns > 0.0
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_probe_cluster_exchange(1792, 16, 1000, 10)
    assert e.value.status == prnn.PRNN_ERR_UNSUPPORTED


# --- dense fp16, wide batches on the tensor cores, K split over clusters of 8 ------------
KSPLIT = [dict(H=2304, B=32, T=24, wdtype="f16", h0_std=0.2),  # 18 clusters, K slices of 288
          dict(H=1152, B=32, T=40, wdtype="f16"),
          dict(H=1152, B=16, T=40, wdtype="f16"),              # N = 32 (hi 16 + lo 16)
          dict(H=1152, B=21, T=20, wdtype="f16", h0_std=0.5),  # odd B: unpadded owner blocks
          dict(H=640, I=200, B=24, T=16, wdtype="f16", h0_std=1.0),  # slices of 80: a half atom
          dict(H=256, B=17, T=30, wdtype="f16"),               # slices of 32
          dict(H=1792, B=20, T=20, wdtype="f16"),
          dict(H=2048, B=16, T=12, wdtype="f16", h0_std=0.3),
          dict(H=128, I=64, B=32, T=50, wdtype="f16"),         # one cluster, one K step
          dict(H=512, B=1, T=20, wdtype="f16", h0_std=0.5),    # N = 16 (hi 8 + lo 8)
          dict(H=384, B=5, T=10, wdtype="f16"),
          dict(H=1024, B=8, T=16, wdtype="f16", h0_std=0.2)]


@pytest.mark.parametrize("spec", KSPLIT)
def test_dense_ksplit_matches_oracle(env, spec):
    """The tensor-core K-split kernel (forced on for every B <= 32; clusters
    of the largest size whose clusters are all resident) stays within the
    rule, and within it of the CUDA-core kernels."""
    _, prnn, o = env
    p = synth.make_problem(seed=105, **spec)
    ref = o.forward(p)
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_KSPLIT: 2},
                      pre_options={prnn.PRNN_OPT_DENSE_KSPLIT: 2})
    cs = info["dense_ksplit"]  # the cluster size
    assert 2 <= cs <= 8 and info["dense_wide_batch"] == 0
    assert info["n_cta"] == p.H // 128 * cs and info["rows_per_cta"] == 128
    check(y, ref, "f16", f"ksplit {spec}")
    y_cc, info_cc = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_KSPLIT: 0})
    assert info_cc["dense_ksplit"] == 0
    assert np.abs(y - y_cc).max() <= TOL["f16"] * float(np.abs(ref).max())


def test_dense_ksplit_exact_properties(env):
    """Determinism, chaining, and batch independence: a column's products do
    not depend on the other columns of its launch (same operand width)."""
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=32, T=16, wdtype="f16", seed=106, h0_std=0.1)
    lay = prnn.Layer.from_problem(p)
    try:
        info = lay.info()
        assert info["dense_ksplit"] == 8 and info["n_cta"] == 72  # the default at B >= 16
        x = torch.from_numpy(p.x).cuda()
        h0 = torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        y_again = lay.forward(x, h0)
        ya = lay.forward(x[:7].contiguous(), h0)
        yb = lay.forward(x[7:].contiguous(), ya[-1].contiguous())
        y20 = lay.forward(x[:, 5:25].contiguous(), h0[5:25].contiguous())
        y16 = lay.forward(x[:, 16:].contiguous(), h0[16:].contiguous())
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    assert torch.equal(y, y_again)
    assert torch.equal(torch.cat([ya, yb]), y)
    assert torch.equal(y20, y[:, 5:25])
    ref = o.forward(p)
    check(y.cpu().numpy(), ref, "f16", "ksplit")
    check(y16.cpu().numpy(), ref[:, 16:], "f16", "ksplit, 16 columns")


def test_dense_ksplit_large_values_are_scaled(env):
    """h of 2^15 or more would overflow the fp16 split: such steps are scaled
    by a power of two first, and the result still follows the oracle."""
    _, prnn, o = env
    p = synth.make_problem(H=512, B=16, T=6, wdtype="f16", seed=107, h0_std=2.0e5)
    ref = o.forward(p)
    assert np.abs(p.h0).max() > 32768.0 and np.abs(ref).max() > 32768.0
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_DENSE_KSPLIT: 2},
                      pre_options={prnn.PRNN_OPT_DENSE_KSPLIT: 2})
    assert info["dense_ksplit"] >= 2
    check(y, ref, "f16", "ksplit, large h")


def test_dense_ksplit_full_size_matches_oracle(env):
    """H = 2304, B = 32 (a sweep point) over the full T = 256, element by
    element against the oracle on every host core."""
    import os
    _, prnn, o = env
    p = synth.make_problem(H=2304, B=32, T=256, wdtype="f16", seed=108)
    y, info = run_gpu(env, p)
    assert info["dense_ksplit"] >= 2 and info["n_cta"] == 18 * info["dense_ksplit"]
    ref = o.forward(p, threads=max(1, os.cpu_count() or 1))
    check(y, ref, "f16", "ksplit full size")


def test_dense_ksplit_default_rule(env):
    """Option 1 (default) runs the K-split kernel where it measured faster
    (H >= 2048 and B >= 4, H >= 1536 and B >= 8, H >= 640 and B >= 12) and
    it is planned (H % 128 == 0, every cluster resident); 0 never; 2 for any B."""
    _, prnn, _ = env
    cases = [(1152, 32, 1), (1152, 16, 1), (1152, 12, 1), (2304, 32, 1), (2304, 8, 1),
             (2304, 4, 1), (1536, 8, 1), (640, 12, 1), (1024, 16, 1), (1152, 8, 0),
             (1024, 8, 0), (2304, 3, 0), (640, 8, 0), (512, 32, 0), (4096, 32, 0),
             (1000, 32, 0)]
    for H, B, want in cases:
        lay = prnn.Layer(H, H, B, "f16", "persistent")
        try:
            p = synth.make_problem(H=H, B=B, T=1, wdtype="f16", seed=109)
            lay.set_problem_weights(p)
            assert (lay.info()["dense_ksplit"] > 0) == want, (H, B)
            lay.set_option(prnn.PRNN_OPT_DENSE_KSPLIT, 0)
            assert lay.info()["dense_ksplit"] == 0
            with pytest.raises(prnn.PrnnError):
                lay.set_option(prnn.PRNN_OPT_DENSE_KSPLIT, 3)
        finally:
            lay.close()


def test_dense_ksplit_times_out_cleanly(env):
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=24, T=6, wdtype="f16", seed=110)
    lay = prnn.Layer.from_problem(p)
    assert lay.info()["dense_ksplit"] == 8
    lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 13)
    lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    lay.forward(torch.from_numpy(p.x).cuda())
    assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    lay.close()
    y, _ = run_gpu(env, p)
    check(y, o.forward(p), "f16", "after timeout")


def test_dense_ksplit_phase_trace(env):
    """The trace build of the K-split kernel gives the same bits, and every
    record names its CTA, cluster size and K slice, with its stamps in step
    order."""
    torch, prnn, o = env
    p = synth.make_problem(H=1152, B=32, T=8, wdtype="f16", seed=111, h0_std=0.2)
    lay = prnn.Layer.from_problem(p)
    try:
        info = lay.info()
        cs, n = info["dense_ksplit"], info["n_cta"]
        assert cs == 8 and n == 72
        x = torch.from_numpy(p.x).cuda()
        h0 = torch.from_numpy(p.h0).cuda()
        y0 = lay.forward(x, h0)
        buf = torch.full((p.T * n * 272,), -1, dtype=torch.int32, device="cuda")
        with pytest.raises(prnn.PrnnError) as e:  # one step short
            prnn.prnn_set_trace_buffer(lay.h, buf, (p.T - 1) * n * 1088)
            lay.forward(x, h0)
        assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
        prnn.prnn_set_trace_buffer(lay.h, buf, buf.numel() * 4)
        y1 = lay.forward(x, h0)
        prnn.prnn_set_trace_buffer(lay.h, None, 0)
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    assert torch.equal(y0, y1)
    check(y1.cpu().numpy(), o.forward(p), "f16", "ksplit traced")
    rec = buf.view(p.T, n, 272)[..., :20].cpu().numpy().view(np.uint32).astype(np.int64)
    assert (rec[..., 1] == np.arange(n)[None, :]).all()
    assert (rec[..., 2] == cs).all() and (rec[..., 3] == np.arange(n)[None, :] % cs).all()
    assert (rec[..., 0] < info["sm_count"]).all()
    steps = rec[..., 4:13]
    gaps = (steps[..., 1:] - steps[..., :-1]) & 0xffffffff
    assert (gaps < (1 << 30)).all()  # each stamp at or after the one before it (mod 2^32)
    issue = (rec[..., 13] - rec[..., 6]) & 0xffffffff
    assert (issue < (1 << 30)).all()  # the MMA issuer's stamp follows the first barrier
    gbar = (rec[..., 15] << 32) | rec[..., 14]
    gpub = (rec[..., 17] << 32) | rec[..., 16]
    assert (gpub > gbar).all() and (gbar[1:].min(axis=1) > gpub[:-1].min(axis=1)).all()


SPARSE_KSPLIT = [dict(H=2304, B=32, T=16, k=576, h0_std=0.2),   # 25 %: the default there
                 dict(H=1152, B=20, T=20, k=115),
                 dict(H=640, I=200, B=17, T=12, k=64, h0_std=0.5),
                 dict(H=256, B=3, T=10, k=20)]


@pytest.mark.parametrize("spec", SPARSE_KSPLIT)
def test_sparse_layer_on_ksplit_matches_oracle(env, spec):
    """A sparse layer's densified matrix on the K-split kernel (forced on)
    stays within the rule and within it of the sparse kernel."""
    _, prnn, o = env
    p = synth.make_problem(seed=112, **spec)
    ref = o.forward(p)
    y, info = run_gpu(env, p, options={prnn.PRNN_OPT_SPARSE_KSPLIT: 2},
                      pre_options={prnn.PRNN_OPT_SPARSE_KSPLIT: 2})
    assert info["sparse"] == 1 and info["dense_ksplit"] >= 2
    check(y, ref, "f16", f"sparse on ksplit {spec}")
    y_sp, info_sp = run_gpu(env, p, options={prnn.PRNN_OPT_SPARSE_KSPLIT: 0},
                            pre_options={prnn.PRNN_OPT_SPARSE_KSPLIT: 0})
    assert info_sp["dense_ksplit"] == 0
    assert np.abs(y - y_sp).max() <= TOL["f16"] * float(np.abs(ref).max())


def test_csr_layer_on_ksplit_matches_oracle(env):
    """An unbalanced (CSR) layer's densified matrix on the K-split kernel."""
    torch, prnn, o = env
    p, _ = synth.make_pruned_pair(H=1152, B=16, T=12, density=0.10, seed=113)
    lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
    try:
        lay.set_option(prnn.PRNN_OPT_SPARSE_KSPLIT, 2)
        lay.set_problem_weights(p)
        assert lay.info()["dense_ksplit"] >= 2
        y = lay.forward(torch.from_numpy(p.x).cuda())
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
    finally:
        lay.close()
    check(y.cpu().numpy(), o.forward(p), "f16", "csr on ksplit")


def test_sparse_ksplit_default_rule(env):
    """Option 1 (default) runs a sparse layer's densified matrix on the
    K-split kernel where the dense rule holds and (entries per row) x B is at
    least 8192 at H >= 1152, 3600 at H >= 1536, 6000 at H >= 2560 (streamed
    weights, B <= 16); 0 never; 3 is refused."""
    _, prnn, _ = env
    cases = [(2304, 0.25, 32, 1), (2304, 0.10, 32, 1), (2304, 0.25, 8, 1), (2048, 0.10, 32, 1),
             (2304, 0.05, 32, 1), (2304, 0.10, 16, 1), (1152, 0.25, 32, 1), (1152, 0.25, 16, 0),
             (1792, 0.10, 16, 0), (2304, 0.05, 16, 0), (2304, 0.10, 8, 0), (2304, 0.25, 4, 0),
             (4096, 0.10, 16, 1), (4096, 0.25, 4, 0), (4096, 0.25, 32, 0)]
    for H, d, B, want in cases:
        p = synth.make_problem(H=H, B=B, T=1, k=synth.sparse_k(H, d), seed=114)
        lay = prnn.Layer(H, H, B, "f16", "persistent")
        try:
            lay.set_problem_weights(p)
            assert (lay.info()["dense_ksplit"] > 0) == bool(want), (H, d, B)
            lay.set_option(prnn.PRNN_OPT_SPARSE_KSPLIT, 0)
            assert lay.info()["dense_ksplit"] == 0
            with pytest.raises(prnn.PrnnError):
                lay.set_option(prnn.PRNN_OPT_SPARSE_KSPLIT, 3)
        finally:
            lay.close()


# --- the K-split kernel with Wh streamed (it does not fit on chip beside the tiles) --------
STREAMED = [dict(H=4096, B=16, T=6, wdtype="f16", h0_std=0.2),   # clusters of 4, slices of 1024
            dict(H=4096, B=11, T=5, wdtype="f16", h0_std=0.5),
            dict(H=4096, I=300, B=4, T=6, wdtype="f16"),          # N = 16 (hi 8 + lo 8)
            dict(H=4096, B=16, T=6, k=1024, h0_std=0.3)]           # a sparse layer, densified


@pytest.mark.parametrize("spec", STREAMED)
def test_ksplit_streamed_matches_oracle(env, spec):
    """H = 4096: the weights stream from their image through each MMA issuer's
    ring of shared-memory stages every step; the result stays within the rule
    and within it of the CUDA-core kernels."""
    _, prnn, o = env
    p = synth.make_problem(seed=115, **spec)
    opts = {prnn.PRNN_OPT_DENSE_KSPLIT: 2, prnn.PRNN_OPT_SPARSE_KSPLIT: 2}
    ref = o.forward(p)
    y, info = run_gpu(env, p, options=opts, pre_options=opts)
    assert info["dense_ksplit"] == 4 and info["n_cta"] == 128
    check(y, ref, "f16", f"streamed {spec}")
    off = {prnn.PRNN_OPT_DENSE_KSPLIT: 0, prnn.PRNN_OPT_SPARSE_KSPLIT: 0}
    y_cc, info_cc = run_gpu(env, p, options=off, pre_options=off)
    assert info_cc["dense_ksplit"] == 0
    assert np.abs(y - y_cc).max() <= TOL["f16"] * float(np.abs(ref).max())


def test_ksplit_streamed_batch_limit_and_timeout(env):
    """The streamed plan serves up to 16 columns (a forward of 32 runs the
    CUDA-core kernel), and a dropped publish ends it in a clean timeout."""
    torch, prnn, o = env
    p = synth.make_problem(H=4096, B=32, T=3, wdtype="f16", seed=116)
    lay = prnn.Layer.from_problem(p)
    try:
        assert lay.info()["dense_ksplit"] == 0
        x = torch.from_numpy(p.x).cuda()
        y32 = lay.forward(x)
        y16 = lay.forward(x[:, :16].contiguous())
        torch.cuda.synchronize()
        assert lay.status() == prnn.PRNN_OK
        lay.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
        lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, 37)
        lay.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 1)
        lay.forward(x[:, :16].contiguous())
        assert lay.status() == prnn.PRNN_ERR_TIMEOUT
    finally:
        lay.close()
    ref = o.forward(p)
    check(y32.cpu().numpy(), ref, "f16", "H=4096 B=32")
    check(y16.cpu().numpy(), ref[:, :16], "f16", "H=4096 B=16 streamed")
