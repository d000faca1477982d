"""CPU tests of the benchmark's multi-rank bookkeeping (replicas only: no
collective on the data path; the slowest rank's time sets the whole-job
value).  Two gloo ranks on 127.0.0.1."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    # per-rank timed seconds: rank 1 is the slow one
    t = bench.max_over_ranks(1.5 + rank, w, "cpu")
    out[rank] = (r, w, lr, t)
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == (0, 2, 0, 2.5) and res[1] == (1, 2, 1, 2.5)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.dist_env()[1] == int(os.environ.get("WORLD_SIZE", 1))


def test_workload_flops():
    import bench
    from persistent_rnn_recurrence_gb300 import synth
    p = synth.named_problem("sparse_f16_h1792_d10_b4_t256", T=2)
    f = bench.workload_flops(p)
    assert f["projection"] == 2.0 * 2 * 4 * 1792 * 1792
    assert f["recurrence"] == 2.0 * 2 * 4 * 1792 * 179


def test_oracle_timing_legs():
    """The CPU-baseline legs: a bounded sample of the workload, the rate
    derived from the timesteps actually run, the host described."""
    import bench
    from persistent_rnn_recurrence_gb300 import synth
    host = bench.host_cpu()
    assert host["cpu_count"] >= 1 and 1 <= host["usable_cores"] <= host["cpu_count"]
    assert isinstance(host["cpu_model"], str) and host["cpu_model"]
    p = synth.named_problem("dense_f32_h256_b4_t32")
    one = bench.time_oracle(p, threads=1, budget=0.2)
    many = bench.time_oracle(p, threads=3, budget=0.2)
    for leg, n in ((one, 1), (many, 3)):
        assert leg["cores"] == n and leg["kind"] == "oracle" and leg["unit"] == "timesteps/s"
        assert leg["seconds"] >= 0.2 and leg["value"] > 0
        runs = int(leg["sample"].split(" run(s)")[0].split(", ")[-1])
        ts = int(leg["sample"].split("first ")[1].split(" of")[0])
        assert ts == p.T   # a sequence this short runs whole, repeated
        assert abs(leg["value"] - runs * ts / leg["seconds"]) <= 1e-9 * leg["value"]


def test_reference_arm_contract():
    """bench.py --impl reference (the fp64 oracle timed on the host cores) prints
    one JSON line with the headline's metric, unit and config and the keys the
    contract names; a rank other than 0 exits 0 without output."""
    import json
    import subprocess
    import sys
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "timesteps/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["dtype"] == "f64"
    assert d["config"]["workload"] == bench.DEFAULT_CONFIG
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert cb["sample"] and cb["host"]["cpu_count"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "timesteps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    env1 = dict(env, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r1 = subprocess.run(cmd, cwd=root, env=env1, capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and not r1.stdout.strip()


def test_traffic_is_null_once_the_kernel_changes(monkeypatch):
    """The DRAM traffic in the bench line comes from the committed capture only
    while the recurrent kernel's sources hash to the captured value."""
    import json
    import bench
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    rec = json.load(open(path))
    key = "sparse_f16_h1792_d10_b4_t256/persistent"
    want = rec[key]["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_sha1", lambda sparse: rec[key]["kernel_source_sha1"])
    assert bench.load_traffic("sparse_f16_h1792_d10_b4_t256", "persistent", True) == want
    monkeypatch.setattr(bench, "kernel_source_sha1", lambda sparse: "0" * 40)
    assert bench.load_traffic("sparse_f16_h1792_d10_b4_t256", "persistent", True) is None
    assert bench.load_traffic("no_such_workload", "persistent", True) is None


def test_sweep_cpu_baseline_leg_checks_parity():
    """The sweep's CPU-baseline leg times the oracle on a point's first steps
    and judges each GPU path's first steps against that output: a path equal
    to the oracle within the rule passes, one with a planted error of 5 % of
    the scale, or a non-finite value, fails."""
    import numpy as np
    import bench
    import oracle
    from persistent_rnn_recurrence_gb300 import synth
    p = synth.make_problem(H=64, B=2, T=40, k=7, seed=3, name="tiny_sweep_point")
    ref = oracle.default().forward(p, T=bench.SWEEP_SAMPLE_T).astype(np.float32)
    bad = ref.copy()
    bad[3, 1, 5] += 0.05 * float(np.abs(ref).max())
    nan = ref.copy()
    nan[0, 0, 0] = np.nan
    out = bench.sweep_cpu_baseline(p, {"persistent": ref, "per_step": ref})
    assert out["parity"]["pass"] and out["parity"]["steps"] == bench.SWEEP_SAMPLE_T
    assert out["cpu_baseline"]["kind"].startswith("oracle") and out["cpu_baseline"]["value"] > 0
    assert not bench.sweep_cpu_baseline(p, {"persistent": ref, "per_step": bad})["parity"]["pass"]
    assert not bench.sweep_cpu_baseline(p, {"persistent": nan, "per_step": ref})["parity"]["pass"]
