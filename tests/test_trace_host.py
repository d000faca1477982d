"""CPU tests of the benchmark's phase-trace analysis: synthetic trace records
with known stamps go through bench.trace_phases (sparse kernel) and
bench.ksplit_trace_phases (dense K-split kernel), and every phase, the step,
the exchange and the publish spread come out as constructed, including
across a wrap of the 32-bit SM clock and with an inactive CTA."""
import numpy as np
import pytest

import bench

WRAP = 1 << 32


def _u32(a):
    return (np.asarray(a, dtype=np.int64) % WRAP).astype(np.uint32)


def _sparse_records(T=4, n=3, nw=2, S=1500, groups=1):
    """[1, T, n, 17, 16] records: CTA n-1 inactive; warp 1 later than warp 0
    by 5 cycles at every stamp after the pass start; SM clocks start 100
    cycles before the 32-bit wrap."""
    off = np.array([0, 40, 60, 700, 780, 1100, 1140, 1230])
    r = np.zeros((1, T, n, 17, 16), dtype=np.int64)
    b0 = WRAP - 100
    for t in range(T):
        for c in range(n):
            r[0, t, c, 0, 1] = c if c < n - 1 else WRAP - 1
            r[0, t, c, 0, 2] = nw
            for w in range(nw):
                s = b0 + t * S + off + np.where(np.arange(8) > 0, 5 * w, 0)
                r[0, t, c, 1 + w, :8] = s
                r[0, t, c, 1 + w, 8] = w                      # re-poll rounds
                g_bar = 10_000 + t * 1000 + c * 10
                g_pub = 10_000 + t * 1000 + 600 + c * 20
                r[0, t, c, 1 + w, 9], r[0, t, c, 1 + w, 10] = g_bar % WRAP, g_bar >> 32
                r[0, t, c, 1 + w, 11], r[0, t, c, 1 + w, 12] = g_pub % WRAP, g_pub >> 32
                r[0, t, c, 1 + w, 13] = s[7] + 30             # record written
    return _u32(r), off, S


def test_sparse_trace_phases_recover_the_stamps():
    rec, off, S = _sparse_records()
    ph = bench.trace_phases(rec, 1000.0)                        # 1 cycle = 1 ns
    T, act = rec.shape[1], 2
    n_samples = (T - 1) * act
    late = 5                                                    # warp 1's lag
    want = {"loop": S + off[0] - off[7] - late,
            "p_request": off[1] + late - off[0]}
    for i, name in enumerate(bench.TRACE_PHASES[2:], start=2):
        want[name] = off[i] - off[i - 1]
    want["step"] = S
    for k, v in want.items():
        assert ph[k].shape == (n_samples,), k
        assert np.all(ph[k] == v), (k, ph[k], v)
    assert np.all(ph["gather_warp"] == off[5] - off[4])
    assert np.all(ph["trace_record_write"] == 30)
    # exchange: this CTA's barrier minus the group's last publish of the step
    # before (CTA 1's, the inactive CTA 2 left out)
    c = np.tile(np.arange(act), T - 1)
    assert sorted(ph["exchange"]) == sorted(400 + 10 * c - 20)
    assert np.all(ph["publish_skew"] == 20)
    assert np.all(ph["rounds"] == 1)
    assert ph["globaltimer_resolution_ns"] == 10.0


def test_sparse_trace_phases_split_by_group():
    rec, _, _ = _sparse_records(n=5)
    rec[:, :, 4, 0, 1] = 4                                      # all five CTAs active
    ph = bench.trace_phases(rec, 1000.0, groups=2)              # CTAs {0, 1}, {2, 3}, {4}
    T = rec.shape[1]
    # per group: barrier of CTA c minus the group's last publish one step before
    want = []
    for grp in ([0, 1], [2, 3], [4]):
        last = 600 + 20 * max(grp)
        want += [1000 + 10 * c - last for _ in range(T - 1) for c in grp]
    assert sorted(ph["exchange"]) == sorted(want)
    assert sorted(ph["publish_skew"]) == sorted([20] * (T - 1) * 2 + [0] * (T - 1))


def test_ksplit_trace_phases_recover_the_stamps():
    T, n, S = 4, 3, 3900
    off = {4: 0, 5: 1170, 6: 1310, 7: 2120, 8: 2520, 9: 2840, 10: 2895, 11: 3175, 12: 3610}
    r = np.zeros((1, T, n, 20), dtype=np.int64)
    b0 = WRAP - 2000
    for t in range(T):
        for c in range(n):
            base = b0 + t * S + 7 * c
            for k, o in off.items():
                r[0, t, c, k] = base + o
            r[0, t, c, 13] = base + off[6] + 760
            g_bar = 50_000 + t * 4000 + c * 32
            g_pub = 50_000 + t * 4000 + 2500 + c * 64
            r[0, t, c, 14], r[0, t, c, 15] = g_bar % WRAP, g_bar >> 32
            r[0, t, c, 16], r[0, t, c, 17] = g_pub % WRAP, g_pub >> 32
            r[0, t, c, 18] = t % 2
    ph = bench.ksplit_trace_phases(_u32(r), 1000.0)
    for name, a, b in bench.KSPLIT_PHASES:
        want = 760 if name == "mma_issue" else off[b] - off[a]
        assert np.all(ph[name] == want), (name, ph[name], want)
        assert ph[name].shape == ((T - 1) * n,)
    assert np.all(ph["step"] == S)
    c = np.tile(np.arange(n), T - 1)
    assert sorted(ph["exchange"]) == sorted(4000 + 32 * c - 2500 - 64 * (n - 1))
    assert np.all(ph["publish_skew"] == 64 * (n - 1))
    assert sorted(ph["rounds"]) == sorted([t % 2 for t in range(1, T) for _ in range(n)])


@pytest.mark.parametrize("mhz", [2070.0, 1000.0])
def test_ksplit_trace_phases_scale_with_the_clock(mhz):
    r = np.zeros((1, 2, 1, 20), dtype=np.int64)
    for t in range(2):
        for k in range(4, 14):
            r[0, t, 0, k] = 1000 * t + 10 * k
    ph = bench.ksplit_trace_phases(_u32(r), mhz)
    assert np.allclose(ph["fill_own"], 10 * 1e3 / mhz)
    assert np.allclose(ph["step"], 1000 * 1e3 / mhz)
