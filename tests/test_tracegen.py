"""The seeded input generator against its own definition.

The generator is shared by the CUDA path's callers and the oracle, so it is
checked here against things fixed outside it: published splitmix64 outputs,
and the composition rules it states (unique indices, carry-over share, the
length each step draws over, the recent window).
"""
import numpy as np
import pytest


def test_splitmix64_published_values(tracegen):
    # splitmix64 from state 0: Vigna's reference generator emits these three first.
    assert tracegen.splitmix64(0) == 0xE220A8397B1DCDAF
    assert tracegen.stream_value(0, 1) == 0x6E789E6AA1B965F4
    assert tracegen.stream_value(0, 2) == 0x06C45D188009454F


def test_zipf_cdf_definition(tracegen):
    cdf = tracegen.zipf_cdf(1.1, 1000)
    ref = np.cumsum((np.arange(1000, dtype=np.float64) + 1.0) ** -1.1)
    assert np.allclose(cdf, ref, rtol=1e-12, atol=0)


@pytest.mark.parametrize("name", ["tiny_b1_c8k", "b32_c32k_s4096", "b256_c32k_grow_tail512"])
def test_rows_follow_recipe(tracegen, name):
    wl = tracegen.WORKLOADS[name]
    steps = min(wl.steps, 24)
    reqs = sorted({0, wl.B - 1})
    tr = tracegen.topk_trace(wl, steps=steps, requests=reqs)
    again = tracegen.topk_trace(wl, steps=steps, requests=reqs, threads=1)
    assert (tr == again).all()  # deterministic, independent of threading
    carry = wl.carry_pct * wl.K // 100
    for i in range(len(reqs)):
        for s in range(steps):
            row = tr[s, i]
            n = wl.len_at(s)
            assert len(np.unique(row)) == wl.K
            assert row.min() >= 0 and row.max() < n
            if s > 0:
                assert len(np.intersect1d(row, tr[s - 1, i])) >= carry
    if len(reqs) > 1:  # request rows differ (keyed by request)
        assert not (tr[:, 0] == tr[:, 1]).all()


def test_recent_window_and_growth(tracegen):
    wl = tracegen.WORKLOADS["b256_c32k_grow_tail512"]
    tr = tracegen.topk_trace(wl, steps=8, requests=[3])
    for s in range(8):
        n = wl.len_at(s)
        assert n == 32769 + s
        assert tr[s, 0].max() < n
    # the newest token is drawable: over many steps some row picks the tail
    assert (tr[:, 0] >= wl.C - wl.T).any()


def test_row_bytes_keyed_by_token(tracegen):
    wl = tracegen.WORKLOADS["tiny_b1_c8k"]
    a = tracegen.rows(wl, 0, 0, 10, 4)
    b = tracegen.rows(wl, 0, 0, 12, 2)
    assert (a[2:] == b).all()
    c = tracegen.rows(wl, 1, 0, 10, 4)
    assert not (a == c).all()
    # roughly uniform bits
    big = tracegen.rows(wl, 0, 0, 0, 512)
    assert abs(np.unpackbits(big).mean() - 0.5) < 0.01


@pytest.mark.parametrize("third", ["zipf", "recent"])
def test_rows_that_take_nearly_every_position(tracegen, third):
    """A row of K indices out of K + 1 positions: once the random draws for one
    index give up, the next free position is taken, so every row is complete,
    distinct and in range (within the recent window for that component)."""
    C, K = 4097, 4096
    kw = dict(third=tracegen.THIRD_ZIPF) if third == "zipf" else dict(third=tracegen.THIRD_RECENT,
                                                                         recent=K)
    # zipf: half carried over, the rest Zipf over every position; recent: every
    # index from the window of the last K positions, which it must fill
    carry = 50 if third == "zipf" else 0
    wl = tracegen.Workload("nearly_full", 47, B=2, C=C, K=K, S=K, T=0, host_ratio=1, layers=1,
                           steps=3, len0=C, grow=0, carry_pct=carry, zipf_pct=0, **kw)
    tr = tracegen.topk_trace(wl, steps=3, requests=[0, 1])
    for s in range(3):
        for i in range(2):
            row = tr[s, i]
            assert len(np.unique(row)) == K
            assert row.min() >= (C - K if third == "recent" else 0) and row.max() < C
