"""Random eviction in the oracle, pinned without the oracle itself: its
generator against SplitMix64's published outputs, its victims against the
invariants of the method, and their spread against a uniform choice."""
import os

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "splitmix64_state0.txt")
GAMMA = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def check_generator(lib):
    want = [int(l, 16) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    # the i-th output from state 0 is one output for the state i * gamma
    got = [lib.or_splitmix64_at((i * GAMMA) & MASK) for i in range(len(want))]
    assert got == want


def _check_invariants(st, before_slot_tok, row, out, counts):
    S = st.S
    # the tables are mutual inverses
    occ = np.nonzero(st.slot_tok >= 0)[0]
    assert np.array_equal(st.tok_slot[st.slot_tok[occ]], occ)
    assert int((st.tok_slot >= 0).sum()) == len(occ)
    # every top-k token is resident, at the slot returned
    valid = row[row >= 0]
    assert np.array_equal(st.slot_tok[out[row >= 0]], valid)
    # the misses are exactly the top-k tokens that were not resident
    was = set(before_slot_tok[before_slot_tok >= 0].tolist())
    assert counts[1] == sum(1 for t in valid.tolist() if t not in was)
    # a slot hit this step keeps its token
    wanted = set(valid.tolist())
    assert all(st.slot_tok[s] == before_slot_tok[s] for s in range(S) if before_slot_tok[s] in wanted)
    # no occupied slot is evicted while an empty one is left unfilled
    evicted = [s for s in range(S) if before_slot_tok[s] >= 0 and st.slot_tok[s] != before_slot_tok[s]]
    if evicted:
        assert int((st.slot_tok < 0).sum()) == 0


def check_invariants(lib, seeds=range(6)):
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        C, S, R, K = 300, 48, 16, 20
        host = np.random.default_rng(seed).integers(0, 256, size=(C, R), dtype=np.uint8)
        st = oracle.RequestState(C, S, 0, R, lib=lib, policy=oracle.POLICY_RANDOM, req=seed, seed=77)
        for step in range(1, 60):
            row = rng.choice(C, size=K, replace=False).astype(np.int32)
            if step % 7 == 0:
                row[::5] = -1
            before = st.slot_tok.copy()
            out, counts, err = st.resolve(host, row, step)
            assert err == 0
            _check_invariants(st, before, row, out, counts)
            # buffer bytes equal the host rows of the resident tokens
            occ = np.nonzero(st.slot_tok >= 0)[0]
            assert np.array_equal(st.buf[occ], host[st.slot_tok[occ]])
            # stamps: the step of last use, as under LRU
            assert np.all(st.stamp[out[row >= 0]] == step)


def _evictions(lib, req, seed, S=64, K=8, steps=2500):
    """Each step asks for K new tokens (all misses, no hits) once the buffer is
    full; returns how often each slot was chosen as a victim."""
    C = S + K * (steps + 2)
    host = np.zeros((C, 16), dtype=np.uint8)
    st = oracle.RequestState(C, S, 0, 16, lib=lib, policy=oracle.POLICY_RANDOM, req=req, seed=seed)
    st.resolve(host, np.arange(S, dtype=np.int32), 1)  # fill every slot
    counts = np.zeros(S, dtype=np.int64)
    nxt = S
    for step in range(2, steps + 2):
        before = st.slot_tok.copy()
        st.resolve(host, np.arange(nxt, nxt + K, dtype=np.int32), step)
        nxt += K
        counts += (st.slot_tok != before)
    return counts


def check_uniform(lib):
    counts = _evictions(lib, req=3, seed=11)
    S, total = len(counts), counts.sum()
    assert total == 8 * 2500
    expected = total / S
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    # 63 degrees of freedom: the 99.99th percentile is about 118
    assert chi2 < 118, chi2
    assert counts.min() > 0


def check_request_and_seed(lib):
    a = _evictions(lib, req=0, seed=5, steps=200)
    assert not np.array_equal(a, _evictions(lib, req=1, seed=5, steps=200))
    assert not np.array_equal(a, _evictions(lib, req=0, seed=6, steps=200))
    assert np.array_equal(a, _evictions(lib, req=0, seed=5, steps=200))  # and on nothing else


def check_random(lib):
    check_generator(lib)
    check_invariants(lib)
    check_uniform(lib)
    check_request_and_seed(lib)


def test_generator_matches_published_outputs():
    check_generator(oracle._lib())


def test_random_eviction_invariants():
    check_invariants(oracle._lib())


def test_random_victims_are_uniform():
    check_uniform(oracle._lib())


def test_random_victims_depend_on_request_and_seed():
    check_request_and_seed(oracle._lib())
