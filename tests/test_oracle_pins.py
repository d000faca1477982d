"""CPU tests: the fp64 oracle against its pins, and the pins' own strength."""
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
from tests import oracle_pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_cells_match_forward(o):
    """The single-output entry the full-size checks use agrees with the
    whole-sequence driver, element for element."""
    from persistent_rnn_recurrence_gb300 import synth
    for p in (synth.make_problem(H=40, B=3, T=3, I=24, wdtype="f32", seed=3, h0_std=0.5),
              synth.make_problem(H=40, B=3, T=3, k=7, seed=4),
              synth.make_pruned_pair(H=40, B=3, T=3, density=0.1, seed=5, row_sigma=1.0)[0]):
        y = o.forward(p)
        samples = [(t, b, r) for t in range(p.T) for b in range(p.B) for r in (0, 17, 39)]
        h0 = np.zeros((p.B, p.H)) if p.h0 is None else p.h0
        got = o.cells(p, samples, lambda t, b: p.x[t, b],
                      lambda t, b: h0[b] if t == 0 else y[t - 1, b])
        want = np.array([y[t, b, r] for (t, b, r) in samples])
        assert np.array_equal(got, want)


def test_delta_cells_match_backward(o):
    """The single-element entry of the reverse recurrence (used by the GPU
    backward checks and the smoke check) agrees with the whole-sequence
    backward, element for element: delta_t[b, r] from dy_t, y_t and
    delta_{t+1} (none at the last step), for dense weights and for a sparse
    layer held densely.  A wrong callback order, a transposed Wh or a
    time-shifted delta_{t+1} in the wrapper fails here."""
    from persistent_rnn_recurrence_gb300 import synth
    for p in (synth.make_problem(H=40, B=3, T=4, I=24, wdtype="f32", seed=11, h0_std=0.5),
              synth.make_problem(H=36, B=2, T=5, k=9, seed=12, h0_std=0.3)):
        dy = np.random.default_rng(13).normal(size=(p.T, p.B, p.H))
        g = o.backward(p, dy)
        d = g["delta"]
        y = o.forward(p)
        if p.sparse:
            Wh = np.zeros((p.H, p.H))
            Wh[np.repeat(np.arange(p.H), p.k), p.cols.astype(np.int64).ravel()] = \
                p.vals.astype(np.float64).ravel()
        else:
            Wh = p.Wh
        samples = [(t, b, r) for t in range(p.T) for b in range(p.B) for r in range(p.H)]
        got = o.delta_cells(Wh, samples, lambda t, b: dy[t, b], lambda t, b: y[t, b],
                            lambda t, b: None if t == p.T - 1 else d[t + 1, b])
        assert np.array_equal(got, d.reshape(-1))
        assert np.count_nonzero(got) > len(samples) // 4   # the check is not vacuous


def test_threaded_driver_gives_the_same_bits(o):
    """The all-cores timing driver splits each step over threads but computes
    every output with the same cell function: the result must be bit-identical
    to the one-thread driver for any team size, including teams larger than
    the number of outputs of a step."""
    from persistent_rnn_recurrence_gb300 import synth
    probs = (synth.make_problem(H=40, B=3, T=5, I=24, wdtype="f32", seed=6, h0_std=0.5),
             synth.make_problem(H=40, B=3, T=5, k=7, seed=7),
             synth.make_problem(H=5, B=1, T=3, I=4, wdtype="f32", seed=8))
    for p in probs:
        y = o.forward(p)
        for n in (1, 2, 3, 8, 64):
            assert np.array_equal(o.forward(p, threads=n), y), (p.H, p.sparse, n)
    p = probs[0]
    with pytest.raises(ValueError):
        o.forward_threads(p.x, p.Wx, p.b, Wh=p.Wh, threads=0)
    with pytest.raises(ValueError):
        o.forward_threads(p.x, p.Wx, p.b, vals=np.ones((40, 1)), cols=np.full((40, 1), 40),
                          threads=2)
    assert o.forward_threads(p.x[:0], p.Wx, p.b, Wh=p.Wh, threads=4).shape == (0, 3, 40)


def test_rejects_bad_arguments(o):
    x = np.zeros((1, 1, 2))
    with pytest.raises(ValueError):
        o.forward_sparse(x, np.zeros((2, 2)), np.ones((2, 1)), np.array([[0], [2]]),
                         np.zeros(2))
    assert o.forward_dense(np.zeros((0, 1, 2)), np.zeros((2, 2)), np.zeros((2, 2)),
                           np.zeros(2)).shape == (0, 1, 2)


# Plausible mistakes, planted in a copy of the oracle's source.  Each must make
# at least one pin fail (the copy runs in a child process).
MUTANTS = {
    "dropped_bias": ("double s = bias[r];", "double s = 0.0;"),
    "transposed_wh": ("Wh[r * H + c]", "Wh[c * H + r]"),
    "transposed_wx": ("Wx[r * I + c] * x_t[c]", "Wx[(c % H) * I + (r % I)] * x_t[c]"),
    "in_place_h": ("y + ((t - 1) * B + b) * H", "y + (t * B + b) * H"),
    "no_relu": ("return s > 0.0 ? s : 0.0;", "return s;"),
    "h0_batch_offset": ("h0 + b * H :", "h0 :"),
    "sparse_wrong_column": ("h_prev[cols[r * k + j]]", "h_prev[j]"),
    "x_batch_index": ("x + (t * B + b) * I", "x + (t * B) * I"),
    "x_time_shift": ("x + (t * B + b) * I", "x + (((t + 1) % T) * B + b) * I"),
    "dropped_recurrent_term": ("s += Wh[r * H + c] * h_prev[c];", "(void)h_prev;"),
    "csr_row_end_off_by_one": ("j < row_ptr[r + 1]; ++j", "j < row_ptr[r + 1] - 1; ++j"),
    "bwd_untransposed_wh": ("g += Wh[c * H + r] * delta_next[c];",
                            "g += Wh[r * H + c] * delta_next[c];"),
    "bwd_no_relu_mask": ("return y_t[r] > 0.0 ? g : 0.0;", "return g;"),
    "bwd_dwh_same_step_h": ("y[((t - 1) * B + b) * H + c];", "y[(t * B + b) * H + c];"),
    "bwd_dx_uses_wh": ("s += Wx[r * I + c] * d[(t * B + b) * H + r];",
                       "s += Wx[(r * I + c) % (H * I)] * d[(t * B + b) * H + (r + 1) % H];"),
    "bwd_dh0_last_delta": ("s += Wh[r * H + c] * d[b * H + r];",
                           "s += Wh[r * H + c] * d[((T - 1) * B + b) * H + r];"),
    "bwd_dwx_time_shift": ("* x[(t * B + b) * I + c];", "* x[(((t + 1) % T) * B + b) * I + c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name} not found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    oracle.compile_oracle(str(mutant), str(lib))
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import oracle\nfrom tests import oracle_pins\n"
            "oracle_pins.run_all(oracle.Oracle(%r))\n") % (ROOT, str(lib))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       cwd=ROOT, timeout=120)
    assert r.returncode != 0, f"mutant {name} passed every pin"


# Plausible mistakes in the Python part of the oracle (the stacking of
# layers), planted in a copy of oracle.py loaded as a separate module.
PY_MUTANTS = {
    "stack_reads_x": ("            inp = y\n", "            inp = x\n"),
    "stack_same_h0": ("None if h0 is None else h0[l]", "None if h0 is None else h0[0]"),
    "stack_reversed": ("enumerate(layers)", "enumerate(layers[::-1])"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_stack_pins_catch_planted_mistake(name):
    import types
    old, new = PY_MUTANTS[name]
    path = os.path.join(ROOT, "oracle", "oracle.py")
    src = open(path).read()
    assert old in src, f"mutation anchor for {name} not found"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = path
    exec(compile(src.replace(old, new), path, "exec"), mod.__dict__)
    o = mod.Oracle(oracle.oracle.LIB)
    with pytest.raises(AssertionError):
        oracle_pins.pin_stack_definition(o)


# Plausible mistakes in the Python wrapper of the reverse-recurrence cell,
# planted in a copy of oracle.py; each must fail the element-for-element
# comparison with the whole-sequence backward.
DELTA_MUTANTS = {
    "dy_and_y_swapped": ("_ptr(_f64(dy_of(t, bb))), _ptr(_f64(y_of(t, bb)))",
                         "_ptr(_f64(y_of(t, bb))), _ptr(_f64(dy_of(t, bb)))"),
    "wh_transposed": ("        Wh = _f64(Wh)\n        H = Wh.shape[0]\n        out = np.zeros(len(samples))",
                      "        Wh = _f64(Wh).T.copy()\n        H = Wh.shape[0]\n        out = np.zeros(len(samples))"),
    "next_delta_dropped": ("None if nx is None else _ptr(_f64(nx))", "None"),
}


@pytest.mark.parametrize("name", sorted(DELTA_MUTANTS))
def test_delta_cells_pin_catches_planted_mistake(name):
    import types
    old, new = DELTA_MUTANTS[name]
    path = os.path.join(ROOT, "oracle", "oracle.py")
    src = open(path).read()
    assert old in src, f"mutation anchor for {name} not found"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = path
    exec(compile(src.replace(old, new), path, "exec"), mod.__dict__)
    with pytest.raises(AssertionError):
        test_delta_cells_match_backward(mod.Oracle(oracle.oracle.LIB))
