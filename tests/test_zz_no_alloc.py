"""GPU tests of prnn_forward_dense_noalloc, the forward entry point for callers
that cannot allocate device memory (code in a latency-critical loop where an
allocation may synchronize the device, or a process whose device memory
belongs to another allocator or a fixed budget).  It uses a fixed scratch
array carried by the library instead of cudaMalloc.

Its output must match the fp64 oracle within the usual rule, and the
handle-based prnn_forward on the same weights, call after call; further calls
must not change the device's free memory; arguments it cannot serve are
refused before anything runs.  This file is collected last so a
stop-at-first-failure run has already run every other test."""
import os

import numpy as np
import pytest

import oracle
from persistent_rnn_recurrence_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2}
SCRATCH_FLOATS = 1 << 22          # the array's size: T*B*H may not exceed it


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    from persistent_rnn_recurrence_gb300 import prnn
    return torch, prnn, oracle.default()


def _device_args(torch, prnn, p):
    wt = torch.float16 if p.wdtype == "f16" else torch.float32
    return dict(
        Wx=torch.from_numpy(p.Wx).cuda().to(wt),
        Wh=torch.from_numpy(p.Wh).cuda().to(wt),
        b=torch.from_numpy(p.b).cuda(),
        x=torch.from_numpy(p.x).cuda(),
        h0=None if p.h0 is None else torch.from_numpy(p.h0).cuda(),
        wd=prnn.PRNN_F16 if p.wdtype == "f16" else prnn.PRNN_F32)


def _call(prnn, p, a, y):
    prnn.prnn_forward_dense_noalloc(p.T, p.B, p.H, p.I, a["wd"], a["x"], a["Wx"], a["Wh"],
                                    a["b"], a["h0"], y)


CASES = [dict(H=256, B=4, T=32, wdtype="f32", h0_std=0.1),
         dict(H=1152, B=4, T=48, wdtype="f16", h0_std=0.1),
         dict(H=300, I=200, B=3, T=7, wdtype="f16"),
         dict(H=301, I=77, B=5, T=9, wdtype="f32", h0_std=0.3),    # H % 4 != 0: scalar loads
         dict(H=4096, B=4, T=256, wdtype="f16")]                   # T*B*H exactly the limit


@pytest.mark.parametrize("spec", CASES, ids=lambda s: f"h{s['H']}_b{s['B']}_t{s['T']}_{s['wdtype']}")
def test_noalloc_matches_oracle_and_handle_forward_twice(env, spec):
    torch, prnn, o = env
    p = synth.make_problem(seed=77, **spec)
    assert p.T * p.B * p.H <= SCRATCH_FLOATS
    a = _device_args(torch, prnn, p)
    ref = o.forward(p, threads=max(1, os.cpu_count() or 1))
    scale = float(np.abs(ref).max())
    assert scale > 0
    # the existing entry point on the same weights (the persistent kernels
    # need H % 4 == 0; the handle's per-step path serves the others)
    lay = prnn.Layer.from_problem(p, algo="persistent" if p.H % 4 == 0 else "per_step")
    y_handle = lay.forward(a["x"], a["h0"])
    torch.cuda.synchronize()
    assert lay.status() == prnn.PRNN_OK
    lay.close()
    for _ in range(2):   # two calls in a row: the shared scratch must not leak state
        y = torch.full_like(y_handle, float("nan"))
        _call(prnn, p, a, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        err = float(np.abs(got - ref).max())
        assert err <= TOL[p.wdtype] * scale, (err, scale)
        err_h = float((y - y_handle).abs().max())
        assert err_h <= TOL[p.wdtype] * scale, (err_h, scale)


def test_noalloc_allocates_nothing(env):
    """After a first call (which may load the library's module on the device),
    further calls leave the device's free memory and the caching allocator's
    reservations unchanged."""
    torch, prnn, _ = env
    p = synth.make_problem(H=1152, B=4, T=64, wdtype="f16", seed=78)
    a = _device_args(torch, prnn, p)
    y = torch.empty(p.T, p.B, p.H, device="cuda")
    _call(prnn, p, a, y)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        _call(prnn, p, a, y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


def test_noalloc_rejects_what_it_cannot_serve(env):
    torch, prnn, _ = env
    p = synth.make_problem(H=256, B=4, T=8, wdtype="f32", seed=79, h0_std=0.1)
    a = _device_args(torch, prnn, p)
    y = torch.full((p.T, p.B, p.H), 7.0, device="cuda")
    spare = torch.zeros(p.T * p.B * p.H + 8, device="cuda")
    wh_spare = torch.zeros(p.H * p.H + 8, device="cuda")
    h0_spare = torch.zeros(p.B * p.H + 8, device="cuda")
    E = prnn.PRNN_ERR_INVALID_ARG

    def refused(T=p.T, B=p.B, H=p.H, I=p.I, wd=a["wd"], x=a["x"], Wx=a["Wx"], Wh=a["Wh"],
                b=a["b"], h0=a["h0"], out=y):
        with pytest.raises(prnn.PrnnError) as e:
            prnn.prnn_forward_dense_noalloc(T, B, H, I, wd, x, Wx, Wh, b, h0, out)
        assert e.value.status == E

    refused(B=33)                                         # more batch columns than served
    refused(T=-1)
    refused(H=0)
    refused(I=0)
    refused(wd=7)                                         # no such weight type
    refused(out=spare[1:].data_ptr())                     # y not 16-byte aligned
    refused(Wh=wh_spare[2:].data_ptr())                   # Wh not 16-byte aligned
    refused(h0=h0_spare[1:].data_ptr())                   # h0 not 16-byte aligned
    refused(x=None)
    refused(T=SCRATCH_FLOATS // (p.B * p.H) + 1)          # beyond the scratch array
    refused(T=64, B=32, H=4096, I=4096)                   # 8 Mi floats > 4 Mi
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())                         # nothing ran
    # T = 0 and B = 0 are no-ops
    prnn.prnn_forward_dense_noalloc(0, p.B, p.H, p.I, a["wd"], a["x"], a["Wx"], a["Wh"], a["b"],
                                    a["h0"], y)
    prnn.prnn_forward_dense_noalloc(p.T, 0, p.H, p.I, a["wd"], a["x"], a["Wx"], a["Wh"], a["b"],
                                    a["h0"], y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
