"""GPU test of prnn_forward_dense_noalloc, the forward entry point for callers
that cannot allocate device memory (it uses a fixed scratch array carried by
the library instead of cudaMalloc).  Its output must match the handle-based
prnn_forward on the same weights, call after call.  This file is collected
last so a stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest

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
    return torch, prnn


@pytest.mark.parametrize("spec", [dict(H=256, B=4, T=32, wdtype="f32", h0_std=0.1),
                                  dict(H=1152, B=4, T=48, wdtype="f16", h0_std=0.1),
                                  dict(H=300, I=200, B=3, T=7, wdtype="f16")])
def test_noalloc_matches_handle_forward_twice(env, spec):
    torch, prnn = env
    p = synth.make_problem(seed=77, **spec)
    wt = torch.float16 if p.wdtype == "f16" else torch.float32
    Wx = torch.from_numpy(p.Wx).cuda().to(wt)
    Wh = torch.from_numpy(p.Wh).cuda().to(wt)
    b = torch.from_numpy(p.b).cuda()
    x = torch.from_numpy(p.x).cuda()
    h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
    wd = prnn.PRNN_F16 if p.wdtype == "f16" else prnn.PRNN_F32
    # reference: the existing entry point (handle, persistent path)
    lay = prnn.Layer.from_problem(p)
    y_ref = lay.forward(x, h0)
    torch.cuda.synchronize()
    assert lay.status() == prnn.PRNN_OK
    lay.close()
    scale = float(y_ref.abs().max())
    for _ in range(2):   # two calls in a row: the shared scratch must not leak state
        y = torch.full_like(y_ref, float("nan"))
        prnn.prnn_forward_dense_noalloc(p.T, p.B, p.H, p.I, wd, x, Wx, Wh, b, h0, y)
        torch.cuda.synchronize()
        err = float((y - y_ref).abs().max())
        assert np.isfinite(err) and err <= TOL[p.wdtype] * scale, (err, scale)


def test_noalloc_rejects_oversized_problem(env):
    torch, prnn = env
    H, B, T = 4096, 32, 64            # T*B*H = 8 Mi floats > the 4 Mi-float scratch
    z = torch.zeros(16, device="cuda")
    with pytest.raises(prnn.PrnnError) as e:
        prnn.prnn_forward_dense_noalloc(T, B, H, H, prnn.PRNN_F16, z, z, z, z, None, z)
    assert e.value.status == prnn.PRNN_ERR_INVALID_ARG
