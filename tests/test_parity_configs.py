"""GPU parity at every named configuration, element by element, against the
fp64 oracle run on all host cores (its threaded driver, which gives the same
bits as the one-thread driver).

Rule, over every output of the compared steps:
    max |y_gpu - y_oracle| <= 2e-2 * max |y_oracle|      (fp16 weights, fp32 accumulation)

* the two large sparse layers (H = 5760, 1 % and 5 % row-balanced, B = 4) over
  the full T = 256, on both recurrent paths;
* the heaviest sweep points over the full T = 256: dense fp16 H = 4096 at
  B = 32 (the largest on-chip layer), row-balanced H = 4096 at 1 % and 25 %
  at B = 16;
* every point of the persistent-versus-per-step sweep (H in {1152, 2304,
  4096}, B in {1, 4, 16, 32}, density in {100, 25, 10, 1} %) over its first
  32 steps, on both paths, in the same launch configuration as the 256-step
  benchmark (the plan does not depend on T).
"""
import os

import numpy as np
import pytest

import oracle
from persistent_rnn_recurrence_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2}
SWEEP_T = 32
ALGOS = ("persistent", "per_step")


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    from persistent_rnn_recurrence_gb300 import prnn
    return torch, prnn, oracle.default()


_REF = {}


def reference(o, p, T):
    """The oracle's y for the first T steps of problem p, on every host core
    (cached: both recurrent paths are compared with the same array)."""
    key = (p.name, p.seed, T)
    if key not in _REF:
        _REF.clear()
        _REF[key] = o.forward(p, T=T, threads=max(1, os.cpu_count() or 1))
    return _REF[key]


def gpu_forward(env, p, algo, T):
    torch, prnn, _ = env
    lay = prnn.Layer.from_problem(p, algo=algo)
    try:
        x = torch.from_numpy(np.ascontiguousarray(p.x[:T])).cuda()
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).cuda()
        y = lay.forward(x, h0)
        st = lay.status()
        assert st == prnn.PRNN_OK, prnn.prnn_status_string(st)
        return y.cpu().numpy()
    finally:
        lay.close()


def check(y, ref, what):
    assert y.shape == ref.shape
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    scale = float(np.abs(ref).max())
    assert scale > 0.0, f"{what}: the reference is all zeros (a vacuous check)"
    err = float(np.abs(y.astype(np.float64) - ref).max())
    assert err <= TOL["f16"] * scale, f"{what}: max err {err:.3e} vs {TOL['f16'] * scale:.3e}"
    # outputs that are exactly zero on one side and not the other can only be
    # ReLU decisions taken on a pre-activation within the rule of 0
    return err / scale


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("name", ["sparse_f16_h5760_d1_b4_t256", "sparse_f16_h5760_d5_b4_t256"])
def test_large_sparse_full_sequence(env, name, algo):
    p = synth.named_problem(name)
    ref = reference(env[2], p, p.T)
    check(gpu_forward(env, p, algo, p.T), ref, f"{name}/{algo}")


def _sweep_problem(name):
    kw = dict(synth.sweep_points())[name]
    return synth.make_problem(name=name, **kw)


HEAVY = ["sweep_h4096_b32_d100", "sweep_h4096_b16_d1", "sweep_h4096_b16_d25"]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("name", HEAVY)
def test_heavy_sweep_points_full_sequence(env, name, algo):
    p = _sweep_problem(name)
    assert p.T == 256
    ref = reference(env[2], p, p.T)
    check(gpu_forward(env, p, algo, p.T), ref, f"{name}/{algo}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("name", [n for n, _ in synth.sweep_points()])
def test_every_sweep_point_first_steps(env, name, algo):
    p = _sweep_problem(name)
    ref = reference(env[2], p, SWEEP_T)
    check(gpu_forward(env, p, algo, SWEEP_T), ref, f"{name}/{algo}")
