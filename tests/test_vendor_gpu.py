"""The per-step vendor-library recurrences that ``bench.py --vendor`` times
(cuBLAS fp32 and fp16 GEMM, cuSPARSE CSR SpMM, each step
h_t = ReLU(P_t + Wh h_{t-1})) and the dense persistent kernel holding a
sparse layer densely compute the same layer as the fp64 oracle: their
outputs are compared element by element, so the persistent-versus-library
ratios of that benchmark rest on checked computations."""
import dataclasses

import numpy as np
import pytest

import oracle
from persistent_rnn_recurrence_gb300 import synth

pytestmark = pytest.mark.gpu

# fp32 loops: x, Wx and Wh are exact in fp32, so only fp32 rounding separates
# them from the oracle; the fp16 GEMM also rounds h and P to fp16 each step
TOL = {"cublas_sgemm": 1e-4, "cusparse_spmm": 1e-4, "cublas_hgemm": 2e-2}


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from persistent_rnn_recurrence_gb300 import build
    build.build()
    import bench
    from persistent_rnn_recurrence_gb300 import prnn
    return torch, bench, prnn, oracle.default()


def _problems():
    yield synth.named_problem("dense_f16_h1152_b4_t256", T=24)
    yield synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=24)
    yield synth.make_problem(H=5760, B=4, T=10, k=57, seed=3303, name="sparse_f16_h5760_d1")
    yield synth.make_pruned_pair(H=300, B=3, T=8, density=0.05, seed=70, row_sigma=1.0)[0]


@pytest.mark.parametrize("i", range(4))
def test_vendor_loops_match_oracle(env, i):
    torch, bench, _, o = env
    p = list(_problems())[i]
    ref = o.forward(p)
    scale = float(np.abs(ref).max())
    assert scale > 0
    loops = bench.vendor_loops(p, torch.device("cuda", 0))
    assert set(loops) >= {"cublas_sgemm", "cublas_hgemm"}
    assert ("cusparse_spmm" in loops) == p.sparse
    for key, (step, P, h0) in loops.items():
        y = bench.vendor_forward(step, P, h0, p.T).cpu().numpy().astype(np.float64)
        err = float(np.abs(y - ref).max())
        assert np.isfinite(y).all() and err <= TOL[key] * scale, (key, err, scale)


@pytest.mark.parametrize("name", ["sparse_f16_h1792_d10_b4_t256", "sparse_f16_h1152_d10"])
def test_sparse_layer_held_densely_matches_oracle(env, name):
    """The benchmark's sparse-versus-dense persistent comparison runs the
    dense persistent kernel on the densified matrix: same layer, same result."""
    torch, bench, prnn, o = env
    if name.startswith("sparse_f16_h1792"):
        p = synth.named_problem(name, T=32)
    else:
        p = synth.make_problem(H=1152, B=4, T=32, k=115, seed=3300, name=name)
    pd = dataclasses.replace(p, Wh=bench.densified_wh(p).astype(np.float16), vals=None,
                             cols=None, name=p.name + "_held_densely")
    lay = prnn.Layer.from_problem(pd)
    try:
        y = lay.forward(torch.from_numpy(p.x).cuda())
        assert lay.status() == prnn.PRNN_OK
        assert lay.info()["sparse"] == 0
    finally:
        lay.close()
    ref = o.forward(p)
    err = float(np.abs(y.cpu().numpy().astype(np.float64) - ref).max())
    assert err <= 2e-2 * float(np.abs(ref).max())
