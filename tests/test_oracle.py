"""Pins of the CPU oracle against things other than itself.

- the hand-worked example in ``golden/hand_example_lru.txt``;
- a brute-force linked-list LRU simulator (``lru_sim.py``) on thousands of
  seeded tiny cases, including errors, padding and a resident tail;
- invariants after every step on synthetic traces;
- closed forms and special cases (cold start, repeated rows, a buffer that
  holds the whole context, no reuse with S = K);
- the qualitative result of the HiSparse blog ("Efficient swap-in kernel"):
  a 4096-slot buffer misses far less than a 2048-slot one under LRU.
"""
import os
import random

import numpy as np
import pytest

from lru_sim import LinkedLRU

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example_lru.txt")


def _host_rows(C, T, R):
    """Host row of token t: every byte equals t (mod 256)."""
    n = C - T
    return (np.arange(n, dtype=np.int64)[:, None] % 256).astype(np.uint8).repeat(R, axis=1)


def _parse_golden():
    cases = []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                parts = line.split()
                kv = dict(p.split("=") for p in parts[2:])
                cur = {"name": parts[1], **{k: int(v) for k, v in kv.items()}, "ops": [], "tail": []}
                cases.append(cur)
            elif line.startswith("tail "):
                cur["tail"] = [int(x) for x in line.split()[1:]]
            elif line == "append":
                cur["ops"].append(("append",))
            elif line.startswith("step "):
                fields = [f.strip() for f in line.split("|")]
                head = fields[0].split()
                step = int(head[1])
                topk = [int(x) for x in head[3:]]
                out = [int(x) for x in fields[1].split()[1:]]
                slot_tok = [int(x) for x in fields[2].split()[1:]]
                stamp = [int(x) for x in fields[3].split()[1:]]
                c = fields[4].split()
                counts = (int(c[1]), int(c[3]), int(c[5]))
                err = int(fields[5].split()[1])
                cur["ops"].append(("step", step, topk, out, slot_tok, stamp, counts, err))
    return cases


def check_golden(oracle_mod, lib=None):
    cases = _parse_golden()
    assert [c["name"] for c in cases] == ["A", "B", "F", "S", "M"]
    R = 16
    for case in cases:
        S, K, C, T, L = case["S"], case["K"], case["C"], case["T"], case["len"]
        sliding = bool(case.get("sliding", 0))
        host = _host_rows(C, T, R)
        st = oracle_mod.RequestState(C, S, T, R, L, lib=lib, policy=case.get("policy", 0),
                                     sliding=sliding)
        tail_rows = {}
        for t in case["tail"]:
            row = np.full(R, 200 + t, dtype=np.uint8)
            st.buf[S + t % T] = row
            tail_rows[t] = row
        step = 0
        for op in case["ops"]:
            if op[0] == "append":
                t = int(st.len[0])
                row = np.full(R, 200 + t, dtype=np.uint8)
                assert st.append(row, host) == 0
                tail_rows[t] = row
                continue
            _, n, topk, out, slot_tok, stamp, counts, err = op
            step += 1
            assert n == step
            assert len(topk) == K
            o, c, e = st.resolve(host, np.array(topk), step, alias=bool(case.get("alias", 0)))
            assert o.tolist() == out, (case["name"], n)
            assert st.slot_tok.tolist() == slot_tok, (case["name"], n)
            assert st.stamp.tolist() == stamp, (case["name"], n)
            assert c == counts, (case["name"], n)
            assert e == err, (case["name"], n)
            # tok_slot is the inverse of slot_tok on occupied entries
            inv = np.full(C, -1, dtype=np.int32)
            for s, t in enumerate(slot_tok):
                if t >= 0:
                    inv[t] = s
            assert st.tok_slot.tolist() == inv.tolist()
            # a token that went through the tail carries its tail bytes (200 + t)
            for s, t in enumerate(slot_tok):
                if t >= 0:
                    assert (st.buf[s] == (200 + t if t in tail_rows else t)).all(), (case["name"], n)
            live = sorted(tail_rows)[-T:] if sliding else sorted(tail_rows)
            for t in live:
                assert (st.buf[S + t % T] == tail_rows[t]).all()
            if sliding:  # written back: every token that left the tail
                for t in sorted(tail_rows)[:-T] if len(tail_rows) > T else []:
                    assert (host[t] == 200 + t).all()


def test_golden_hand_example(oracle_lib):
    check_golden(oracle_lib)


def _random_case(rng):
    S = rng.randint(1, 12)
    K = rng.randint(1, S)
    T = 0 if rng.random() < 0.6 else rng.randint(1, 6)
    cold = rng.randint(max(K, 1), 40)
    C = cold + T
    grow = T > 0 and rng.random() < 0.5
    length = C - T if grow else C
    steps = rng.randint(1, 25)
    return S, K, T, C, length, grow, steps


def _random_row(rng, K, length, prev, p_bad):
    row = []
    pool = list(range(length))
    rng.shuffle(pool)
    carry = [t for t in (prev or []) if 0 <= t < length]
    rng.shuffle(carry)
    ncarry = rng.randint(0, min(len(carry), K)) if carry else 0
    row = carry[:ncarry]
    for t in pool:
        if len(row) >= K:
            break
        if t not in row:
            row.append(t)
    while len(row) < K:
        row.append(-1)
    rng.shuffle(row)
    if rng.random() < p_bad:
        j = rng.randrange(K)
        kind = rng.randrange(4)
        if kind == 0:
            row[j] = -1
        elif kind == 1:
            row[j] = length + rng.randrange(3)
        elif kind == 2:
            row[j] = -2 - rng.randrange(3)
        elif K > 1:
            row[j] = row[(j + 1) % K]
    return row


def check_against_simulator(oracle_mod, seeds, lib=None, fifo=False, sliding=False, alias=False):
    R = 8
    for seed in seeds:
        rng = random.Random(seed)
        S, K, T, C, length, grow, steps = _random_case(rng)
        if sliding:
            if T == 0:
                T = rng.randint(1, 6)
                C += T
            grow, length = True, rng.randint(0, C - 1)
        host = _host_rows(C, T, R)
        host_sim = host.copy()
        st = oracle_mod.RequestState(C, S, T, R, length, lib=lib, policy=1 if fifo else 0,
                                     sliding=sliding)
        sim = LinkedLRU(S, T, C, length, host_row=lambda t: host_sim[t].copy(), fifo=fifo,
                        sliding=sliding, host_store=host_sim, alias=alias)
        if sliding:  # the tail starts with the last T tokens written
            for t in range(max(0, length - T), length):
                row = np.full(R, (150 + t) % 256, dtype=np.uint8)
                st.buf[S + t % T] = row
                sim.buf[S + t % T] = row.copy()
        prev = None
        for s in range(1, steps + 1):
            if grow and rng.random() < 0.7:
                row_bytes = np.full(R, 100 + (st.len[0] % 100), dtype=np.uint8)
                e1 = st.append(row_bytes, host)
                e2 = sim.append(row_bytes)
                assert (e1 != 0) == (e2 != 0)
            topk = _random_row(rng, K, int(st.len[0]), prev, p_bad=0.15)
            if alias and K > 1:  # a second position repeating some of the first's tokens
                half = K // 2
                topk = topk[:half] + [topk[rng.randrange(half)] if rng.random() < 0.4 else t
                                      for t in topk[half:]]
            prev = topk
            o, c, e = st.resolve(host, np.array(topk), s, alias=alias)
            so, sc, se = sim.step(topk)
            ctx = (seed, s)
            assert o.tolist() == so, ctx
            assert c == sc, ctx
            assert e == se, ctx
            assert st.slot_tok.tolist() == [(-1 if x is None else x) for x in sim.content], ctx
            # recency: the oracle's (stamp, slot) order is the simulator's list order
            order = sorted(range(S), key=lambda i: (int(st.stamp[i]), i))
            assert order == sim.order(), ctx
            for v in range(S + T):
                if sim.buf[v] is not None:
                    assert (st.buf[v] == sim.buf[v]).all(), ctx


@pytest.mark.parametrize("seed_block", range(4))
def test_oracle_matches_linked_list_lru(oracle_lib, seed_block):
    check_against_simulator(oracle_lib, range(seed_block * 600, (seed_block + 1) * 600))


def test_oracle_sliding_tail_matches_linked_list(oracle_lib):
    """Sliding tail: tokens leave the tail into their host rows."""
    check_against_simulator(oracle_lib, range(7000, 7800), sliding=True)
    check_against_simulator(oracle_lib, range(8000, 8300), sliding=True, fifo=True)


def test_oracle_alias_matches_linked_list(oracle_lib):
    """Several positions in one step: repeats share their first occurrence's slot."""
    check_against_simulator(oracle_lib, range(9000, 9800), alias=True)


def test_oracle_fifo_matches_linked_list(oracle_lib):
    """FIFO: only refills move a slot in the recency order."""
    check_against_simulator(oracle_lib, range(5000, 5800), fifo=True)


def test_lru_beats_fifo_on_reuse(oracle_lib, tracegen):
    """The pages' comparison of eviction strategies: on a trace with reuse,
    LRU misses less than FIFO at the same buffer size.  (With S = K every slot
    is hit or refilled each step and the two policies coincide, so this uses
    the 4096-slot buffer.)"""
    wl = tracegen.WORKLOADS["b64_c64k_s4096"]
    tr = tracegen.topk_trace(wl, steps=30, requests=[0, 1])
    tot = {}
    for policy in (0, 1):
        m = 0
        for i in range(2):
            host = np.zeros((wl.cold, 16), np.uint8)
            _, _, counts, _ = oracle_lib.run_request(wl.C, wl.S, wl.T, 16, host, tr[:, i],
                                                     policy=policy)
            m += counts[10:, 1].sum()
        tot[policy] = m
    assert tot[0] < tot[1]


def _check_invariants(st, topk, out, step, host, S, T, C):
    occ = st.slot_tok >= 0
    # slot maps are mutual inverses on occupied entries
    toks = st.slot_tok[occ]
    assert (st.tok_slot[toks] == np.nonzero(occ)[0]).all()
    assert (st.tok_slot >= 0).sum() == occ.sum()
    # every cold top-k token is resident, with its stamp at this step
    cold = (topk >= 0) & (topk < C - T)
    assert (st.tok_slot[topk[cold]] == out[cold]).all()
    assert (st.stamp[out[cold]] == step).all()
    # every other stamp is older
    others = np.ones(S, dtype=bool)
    others[out[cold]] = False
    assert (st.stamp[others] < step).all()
    # buffer bytes equal the host rows of the resident tokens
    assert (st.buf[:S][occ] == host[toks]).all()


def test_oracle_invariants_on_synthetic_trace(oracle_lib, tracegen):
    for name in ("tiny_b1_c8k",):
        wl = tracegen.WORKLOADS[name]
        tr = tracegen.topk_trace(wl)
        host = tracegen.rows(wl, 0, 0, 0, wl.cold)
        st = oracle_lib.RequestState(wl.C, wl.S, wl.T, wl.row_bytes)
        occupied = 0
        for s in range(wl.steps):
            topk = tr[s, 0]
            resident_before = set(np.nonzero(st.tok_slot >= 0)[0].tolist())
            out, (h, m, ip), e = st.resolve(host, topk, s + 1)
            assert e == 0
            # miss count = |top-k \ resident set before the step|
            assert m == len(set(topk.tolist()) - resident_before)
            assert h + m + ip == wl.K
            _check_invariants(st, topk, out, s + 1, host, wl.S, wl.T, wl.C)
            occ_now = int((st.slot_tok >= 0).sum())
            assert occupied <= occ_now <= wl.S
            occupied = occ_now
            if s == 0:
                assert m == wl.K  # cold start: every index misses


def test_oracle_special_cases(oracle_lib):
    R = 4
    rng = np.random.default_rng(7)
    # (a) a step that repeats the previous row misses nothing
    C, S, K = 64, 16, 8
    host = _host_rows(C, 0, R)
    st = oracle_lib.RequestState(C, S, 0, R)
    row = rng.choice(C, K, replace=False).astype(np.int32)
    _, (h, m, _), _ = st.resolve(host, row, 1)
    assert (h, m) == (0, K)
    out1 = None
    for s in range(2, 6):
        out, (h, m, _), _ = st.resolve(host, rng.permutation(row), s)
        assert (h, m) == (K, 0)
    # (b) S >= C: misses are exactly the first touches
    C, S, K = 24, 24, 6
    host = _host_rows(C, 0, R)
    st = oracle_lib.RequestState(C, S, 0, R)
    seen = set()
    for s in range(1, 30):
        row = rng.choice(C, K, replace=False).astype(np.int32)
        _, (h, m, _), _ = st.resolve(host, row, s)
        new = set(row.tolist()) - seen
        assert m == len(new) and h == K - len(new)
        seen |= new
    # (c) S = K and no reuse: every index misses and every slot is a victim
    C, S, K = 200, 10, 10
    host = _host_rows(C, 0, R)
    st = oracle_lib.RequestState(C, S, 0, R)
    for s in range(1, 21):
        row = np.arange((s - 1) * K, s * K, dtype=np.int32)[::-1].copy()
        out, (h, m, _), _ = st.resolve(host, row, s)
        assert (h, m) == (0, K)
        assert sorted(out.tolist()) == list(range(S))
        # pairing: i-th miss in row order takes the i-th lowest slot
        assert out.tolist() == list(range(S))
        assert (st.stamp == s).all()
    # (d) an all-padding row changes nothing
    before = (st.tok_slot.copy(), st.slot_tok.copy(), st.stamp.copy())
    out, c, e = st.resolve(host, np.full(K, -1, dtype=np.int32), 21)
    assert (out == -1).all() and c == (0, 0, 0) and e == 0
    assert all((a == b).all() for a, b in zip(before, (st.tok_slot, st.slot_tok, st.stamp)))
    # (e) errors leave the state untouched
    out, c, e = st.resolve(host, np.array([C, -5, 3, 3], dtype=np.int32), 22)
    assert e == 3 and out.tolist()[:2] == [-1, -1] and out[3] == -1 and out[2] >= 0


def test_larger_buffer_misses_less(oracle_lib, tracegen):
    """HiSparse blog, "Efficient swap-in kernel": 4096 LRU slots miss far less than 2048."""
    w4 = tracegen.WORKLOADS["b64_c64k_s4096"]
    w2 = tracegen.WORKLOADS["b64_c64k_s2048"]
    steps, reqs = 40, [0, 1, 2, 3]
    tr = tracegen.topk_trace(w4, steps=steps, requests=reqs)
    tr2 = tracegen.topk_trace(w2, steps=steps, requests=reqs)
    assert (tr == tr2).all()  # the sweep uses one trace
    tot = {}
    for wl in (w4, w2):
        m = 0
        for i, b in enumerate(reqs):
            host = tracegen.rows(wl, 0, b, 0, wl.cold)
            _, _, counts, errs = oracle_lib.run_request(wl.C, wl.S, wl.T, wl.row_bytes, host, tr[:, i])
            assert (errs == 0).all()
            assert counts[0, 1] == wl.K
            m += counts[10:, 1].sum()
        tot[wl.S] = m
    assert tot[4096] < 0.9 * tot[2048]
