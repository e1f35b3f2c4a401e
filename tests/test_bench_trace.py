"""The step trace's host side (bench.py --trace): launches split where the
kernel kind changes, and the per-boundary intervals of a synthetic step whose
timestamps are laid out by hand, so that every interval has a known value."""
import numpy as np
import pytest


def _recs(rows):
    import bench
    r = np.zeros(len(rows), dtype=np.dtype(bench.TRACE_DTYPE))
    for i, (kind, cta, t) in enumerate(rows):
        r[i]["kind"] = kind
        r[i]["cta"] = cta
        r[i]["t"] = t
    return r


def _product(kind, t0, n=4):
    # start, producer wait, consumers' wait, first stage, loop done, end (ns);
    # CTA c's loop ends c * 100 ns after CTA 0's
    return [(kind, c, [t0, t0 + 500, t0 + 1000, t0 + 2000, t0 + 10000 + 100 * c, t0 + 10000 + 100 * c + 50])
            for c in range(n)]


def _prep(kind, t0, n=4):
    # start, wait returned, loads done, statistics, stores, end
    return [(kind, c, [t0, t0 + 1000, t0 + 3000, t0 + 3600, t0 + 4600, t0 + 4700]) for c in range(n)]


def test_launches_split_where_the_kind_changes():
    import bench
    rows = _prep(3001, 0, 1) + _product(1101, 100) + _prep(2400, 11000) + _product(1121, 16000)
    segs = bench.trace_launches(_recs(rows))
    assert [k for k, _ in segs] == [3001, 1101, 2400, 1121]
    assert [len(i) for _, i in segs] == [1, 4, 4, 4]


def test_dense_boundary_intervals():
    import bench
    # prep 0 (x0), product A (1101), prep 1 (2400), product B (1121), prep 2 (2410), product C (1101)
    rows = (_prep(3001, 0, 1) + _product(1101, 1000) + _prep(2400, 11000) + _product(1121, 16000)
            + _prep(2410, 27000) + _product(1101, 32000))
    s = bench.trace_summary_dense(_recs(rows))
    a = s["by_product_kind_us"]["1101"]
    assert a["launches"] == 1          # the last product has no boundary after it
    assert a["wait->first stage"] == pytest.approx(1.0)
    # median loop end 1000 + 10150, first stage at 3000: 8.15 us
    assert a["stream (median CTA)"] == pytest.approx(8.15)
    assert a["CTA spread"] == pytest.approx(0.15)               # 10300 - 10150
    # last CTA ends at 1000 + 10350; prep 1 waits from 12000
    assert a["last CTA -> prep wait"] == pytest.approx(0.65)
    assert a["prep loads"] == pytest.approx(2.0)
    assert a["prep statistics barrier"] == pytest.approx(0.6)
    assert a["prep bands and stores"] == pytest.approx(1.0)
    # prep 1 ends at 15700, product B's consumers wait until 17000
    assert a["prep end -> next wait"] == pytest.approx(1.3)
    assert a["next wait -> first stage"] == pytest.approx(1.0)
    assert s["by_product_kind_us"]["1121"]["launches"] == 1
    assert s["span_us"] == pytest.approx((32000 + 10350) / 1e3, abs=0.05)   # rounded to 0.1 us


def test_moe_layer_intervals():
    import bench
    rows = []
    t = 0
    for _ in range(3):   # three MoE layers: prep, gate/up, h prep, down
        rows += _prep(3104, t)
        rows += _product(4031, t + 5000)
        rows += _prep(3001, t + 16000)
        rows += _product(4011, t + 21000)
        t += 32000
    rows += _prep(3104, t)
    s = bench.trace_summary_moe(_recs(rows))
    assert s["moe_layers"] == 2        # a layer needs the kernel before it and the prep after it
    lay = s["per_layer_us"]
    assert lay["layer"] == pytest.approx(32.0)
    assert lay["MoE prep"] == pytest.approx(3.7)
    assert lay["gate/up stream (median CTA)"] == pytest.approx(8.15)
    assert lay["h prep"] == pytest.approx(3.7)
    # down ends at 21000 + 10350; the next prep waits from 32000 + 1000
    assert lay["-> next prep wait"] == pytest.approx(1.65)
