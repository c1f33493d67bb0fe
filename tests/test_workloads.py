"""Host checks of the seeded workload recipes (no GPU): group-size readings of
the pages' vocabulary and the table of the pages' GB300 rows."""
import numpy as np
import pytest

from moe_ragged_grouped_gb300 import workloads as wl


def test_zipf_one_empty_matches_skewed_config():
    # the skewed configuration's sizes: Zipf(1.2) over three groups, one empty group first
    assert wl.zipf_sizes(4, 136064, 1.2, one_empty=True, ascending=True) == [0, 21381, 34780, 79903]
    assert wl.zipf_sizes_one_empty(4, 136064, 1.2) == [0, 21381, 34780, 79903]


@pytest.mark.parametrize("E,M", [(4, 112576), (4, 136064), (8, 131072), (32, 131072)])
@pytest.mark.parametrize("one_empty", [False, True])
def test_zipf_sizes_sum_order_and_ratios(E, M, one_empty):
    d = wl.zipf_sizes(E, M, 1.2, one_empty=one_empty)
    a = wl.zipf_sizes(E, M, 1.2, one_empty=one_empty, ascending=True)
    assert sum(d) == M and len(d) == E and a == d[::-1]
    assert d == sorted(d, reverse=True)
    assert (d[-1] == 0) == one_empty
    nz = np.array([v for v in d if v > 0], np.float64)
    # consecutive groups follow i^-1.2 up to the integer rounding
    want = np.array([(i + 1) ** -1.2 for i in range(len(nz))])
    assert np.allclose(nz / nz.sum(), want / want.sum(), atol=2.0 / M)


def test_lognormal_sizes_are_seeded_and_sum_to_M():
    s1 = wl.lognormal_sizes(16, 131072, 0.35, 0)
    assert s1 == wl.lognormal_sizes(16, 131072, 0.35, 0) and sum(s1) == 131072
    cv = np.std(s1) / np.mean(s1)
    assert 0.15 < cv < 0.6


def test_pages_rows_parse():
    assert len(wl.PAGES_GB300_ROWS) == 100
    ops = [r[1] for r in wl.PAGES_GB300_ROWS]
    assert ops.count("dW") == 36 and ops.count("ckpt") == 32 and ops.count("ckpt ES") == 32
    for shape, op, det_ms, sota_ms, key, nd_ms in wl.PAGES_GB300_ROWS:
        wk, od = wl.pages_workload(shape)
        assert wk.M == int(shape.split()[2][1:]) and sum(wk.sizes) == wk.M
        assert (wk.N, wk.K) == wl.PAGES_SHAPES[shape.split()[0]]
        assert od == ("fp32" if shape.endswith("fp32") else "bf16")
        assert det_ms > 0 and sota_ms > 0 and nd_ms > 0 and key in "tcd"
        # derived throughput of the pages' own numbers lies below the dense peak
        assert wk.flops(len(wl.PAGES_OPS[op])) / (det_ms * 1e-3) < 2.25e15
