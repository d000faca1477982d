"""GPU parity of stacked layers (prnn_stack_*): both the one-launch wavefront
and the layer-by-layer path against the fp64 oracle, through the C ABI.

Rule per layer, over the whole sequence:
    max |y_gpu[l] - y_oracle[l]| <= tol * max |y_oracle[l]|
with tol = 1e-4 for fp32 weights and 2e-2 for fp16 weights.
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


def run_stack(env, p, algo, options=None):
    torch, prnn, _ = env
    st = prnn.Stack.from_problem(p, algo=algo)
    try:
        for k, v in (options or {}).items():
            st.set_option(k, v)
        x = torch.from_numpy(p.x).cuda()
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
        y = st.forward(x, h0)
        s = st.status()
        assert s == prnn.PRNN_OK, prnn.prnn_status_string(s)
        return y.cpu().numpy(), st.info()
    finally:
        st.close()


def check_layers(y, ref, wdtype, what):
    assert y.shape == ref.shape
    assert np.isfinite(y).all(), what
    for l in range(ref.shape[0]):
        scale = float(np.abs(ref[l]).max())
        err = float(np.abs(y[l].astype(np.float64) - ref[l]).max())
        assert err <= TOL[wdtype] * scale, f"{what} layer {l}: {err:.3e} vs {TOL[wdtype] * scale:.3e}"


CASES = [
    dict(L=2, H=256, I=128, B=3, T=6, wdtype="f32", h0_std=0.5),
    dict(L=3, H=1152, B=4, T=32, wdtype="f16"),
    dict(L=4, H=512, B=4, T=16, wdtype="f16", h0_std=0.2),
    dict(L=2, H=300, I=100, B=5, T=7, wdtype="f16"),
    dict(L=8, H=256, B=2, T=10, wdtype="f16"),
    dict(L=2, H=1152, B=1, T=20, wdtype="f16"),
    dict(L=1, H=640, B=32, T=4, wdtype="f16"),
    dict(L=2, H=8, I=4, B=2, T=3, wdtype="f32", h0_std=1.0),
]


@pytest.mark.parametrize("algo", ["wavefront", "layerwise"])
@pytest.mark.parametrize("i", range(len(CASES)))
def test_stack_matches_oracle(env, i, algo):
    p = synth.make_stack_problem(seed=400 + i, **CASES[i])
    y, info = run_stack(env, p, algo)
    assert info["layers_set"] == p.L
    check_layers(y, env[2].forward(p), p.wdtype, f"case{i}/{algo}")


def test_stack_full_size_two_layers(env):
    """Two H = 1152 fp16 layers over the full 256 steps, both paths."""
    p = synth.make_stack_problem(L=2, H=1152, B=4, T=256, wdtype="f16", seed=420, h0_std=0.1)
    ref = env[2].forward(p)
    for algo in ("wavefront", "layerwise"):
        y, info = run_stack(env, p, algo)
        check_layers(y, ref, "f16", algo)
        if algo == "wavefront":
            assert info["n_cta_per_layer"] * p.L <= 152 * 2


def test_stack_wavefront_deterministic_and_chains(env):
    """Bit-identical reruns; running steps [0, T1) then [T1, T) from the last
    outputs (h0 = y[:, T1-1]) equals one run over [0, T)."""
    torch, prnn, _ = env
    p = synth.make_stack_problem(L=3, H=512, B=4, T=12, wdtype="f16", seed=421, h0_std=0.3)
    st = prnn.Stack.from_problem(p)
    try:
        x = torch.from_numpy(p.x).cuda()
        h0 = torch.from_numpy(p.h0).cuda()
        ya = st.forward(x, h0).clone()
        yb = st.forward(x, h0).clone()
        assert torch.equal(ya, yb)
        y1 = st.forward(x[:5].contiguous(), h0).clone()
        y2 = st.forward(x[5:].contiguous(), y1[:, -1].contiguous()).clone()
        assert torch.equal(torch.cat([y1, y2], dim=1), ya)
        assert st.status() == prnn.PRNN_OK
    finally:
        st.close()


def test_stack_forced_groups(env):
    torch, prnn, o = env
    p = synth.make_stack_problem(L=2, H=256, B=4, T=8, wdtype="f16", seed=422)
    ref = o.forward(p)
    for g in (1, 2, 4):
        st = prnn.Stack(p.L, p.H, p.I, p.B, "f16", "wavefront")
        try:
            st.set_option(prnn.PRNN_OPT_CTA_GROUPS, g)
            st.set_problem_weights(p)
            assert st.info()["cta_groups"] == g
            y = st.forward(torch.from_numpy(p.x).cuda())
            assert st.status() == prnn.PRNN_OK
            check_layers(y.cpu().numpy(), ref, "f16", f"G={g}")
        finally:
            st.close()


def test_stack_errors(env):
    torch, prnn, _ = env
    with pytest.raises(prnn.PrnnError) as e:                  # hidden not a multiple of 4
        prnn.prnn_stack_create(2, 130, 128, 4, prnn.PRNN_F16, prnn.PRNN_STACK_WAVEFRONT)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    with pytest.raises(prnn.PrnnError) as e:                  # too many layers
        prnn.prnn_stack_create(9, 128, 128, 4, prnn.PRNN_F16, prnn.PRNN_STACK_WAVEFRONT)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    with pytest.raises(prnn.PrnnError) as e:                  # weights cannot all be on chip
        prnn.prnn_stack_create(8, 4096, 4096, 4, prnn.PRNN_F16, prnn.PRNN_STACK_WAVEFRONT)
    assert e.value.status == prnn.PRNN_ERR_UNSUPPORTED
    p = synth.make_stack_problem(L=2, H=64, B=2, T=3, wdtype="f16", seed=423)
    s = prnn.prnn_stack_create(2, 64, 64, 2, prnn.PRNN_F16, prnn.PRNN_STACK_WAVEFRONT)
    x = torch.from_numpy(p.x).cuda()
    y = torch.empty(2, 3, 2, 64, device="cuda")
    Wx, Wh, b = (torch.from_numpy(a).cuda() for a in p.layers[0])
    prnn.prnn_stack_set_layer(s, 0, Wx, Wh, b)
    with pytest.raises(prnn.PrnnError) as e:                  # layer 1 not set
        prnn.prnn_stack_forward(s, 3, 2, x, None, y)
    assert e.value.status == prnn.PRNN_ERR_NOT_READY
    Wx, Wh, b = (torch.from_numpy(a).cuda() for a in p.layers[1])
    prnn.prnn_stack_set_layer(s, 1, Wx, Wh, b)
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_stack_set_layer(s, 2, Wx, Wh, b)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    with pytest.raises(prnn.PrnnError) as e:                  # y overlaps x
        prnn.prnn_stack_forward(s, 3, 2, x, None, x)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    with pytest.raises(prnn.PrnnError) as e:                  # B > max_batch
        prnn.prnn_stack_forward(s, 3, 3, x, None, y)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
    prnn.prnn_stack_forward(s, 0, 2, x, None, y)              # no-ops
    prnn.prnn_stack_forward(s, 3, 0, x, None, y)
    prnn.prnn_stack_forward(s, 3, 2, x, None, y)
    assert prnn.prnn_stack_get_status(s) == prnn.PRNN_OK
    prnn.prnn_stack_destroy(s)


def test_stack_dropped_publish_times_out_cleanly(env):
    """A CTA of the second layer's slice skips one publish: the third layer
    and the second layer's next step wait for it; the launch ends with a
    TIMEOUT status (sticky), and a fresh stack then computes correctly."""
    torch, prnn, o = env
    p = synth.make_stack_problem(L=3, H=256, B=4, T=6, wdtype="f16", seed=424)
    st = prnn.Stack.from_problem(p)
    n = st.info()["n_cta_per_layer"]
    st.set_option(prnn.PRNN_OPT_WAIT_TIMEOUT_US, 20000)
    st.set_option(prnn.PRNN_OPT_DEBUG_DROP_CTA, n + 1)
    st.set_option(prnn.PRNN_OPT_DEBUG_DROP_STEP, 2)
    x = torch.from_numpy(p.x).cuda()
    st.forward(x)
    assert st.status() == prnn.PRNN_ERR_TIMEOUT
    with pytest.raises(prnn.PrnnError) as e:
        st.forward(x)
    assert e.value.status == prnn.PRNN_ERR_TIMEOUT
    st.close()
    y, _ = run_stack(env, p, "wavefront")
    check_layers(y, o.forward(p), "f16", "after timeout")


def test_layerwise_stack_at_wide_batch(env):
    """A layer-by-layer stack at a wide batch: each dense fp16 layer's
    forward runs the tensor-core K-split kernel (the single-layer default at
    H=1152, B=16), and every layer matches the oracle."""
    _, _, o = env
    p = synth.make_stack_problem(L=2, H=1152, B=16, T=10, wdtype="f16", seed=425, h0_std=0.2)
    y, _ = run_stack(env, p, "layerwise")
    check_layers(y, o.forward(p), "f16", "layerwise stack, wide batch")
