"""Resuming from an imported state, and LRU selection among old stamps.

hs_import_state loads tables and stamps saved earlier (hs_export_state's
layout).  The tests start the GPU and the oracle from the same randomised
state at a large step count, so that the victim search runs through every
branch of its age histogram: the m-th oldest slot in an exact age bin, or
among the ages >= 1023 (then a radix select over 1, 2, 3 or 4 stamp digits).
Results are compared exactly with the oracle, in both launch modes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_all()
    import oracle
    oracle.build()


def _random_state(rng, C, S, cold, step0, old_frac, occupancy=1.0):
    tok_slot = np.full(C, -1, dtype=np.int32)
    slot_tok = np.full(S, -1, dtype=np.int32)
    stamp = np.zeros(S, dtype=np.int32)
    occ = rng.choice(S, size=int(occupancy * S), replace=False)
    toks = rng.choice(cold, size=len(occ), replace=False).astype(np.int32)
    slot_tok[occ] = toks
    tok_slot[toks] = occ
    old = rng.random(len(occ)) < old_frac
    lim = max(step0 - 1023, 0)
    stamp[occ] = np.where(old, rng.integers(0, lim + 1, len(occ)),
                          rng.integers(lim, step0 + 1, len(occ))).astype(np.int32)
    return tok_slot, slot_tok, stamp


def _rows(rng, st_tok_slot, cold, C, K, hit_frac):
    resident = np.nonzero(st_tok_slot >= 0)[0]
    nh = min(int(hit_frac * K), len(resident))
    hits = rng.choice(resident, size=nh, replace=False)
    pool = np.setdiff1d(np.arange(C), hits)
    new = rng.choice(pool, size=K - nh, replace=False)
    row = np.concatenate([hits, new]).astype(np.int32)
    rng.shuffle(row)
    return row


@pytest.mark.parametrize("policy", [0, 1], ids=["lru", "fifo"])
@pytest.mark.parametrize("mode", [1, 2, 3], ids=["fused", "split", "cluster"])
@pytest.mark.parametrize("step0,old_frac", [(5000, 0.5), (5000, 0.03), (100000, 0.6),
                                            ((1 << 30) + 12345, 0.7), (700, 0.5)])
def test_resume_matches_oracle(mode, step0, old_frac, policy):
    import oracle
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg

    B, C, K, S, T, R, ratio = 6, 20000, 1024, 2048, 0, 1152, 10
    wl = tg.Workload("resume", 99, B=B, C=C, K=K, S=S, T=T, host_ratio=ratio, layers=1, steps=1,
                     len0=C, grow=0, carry_pct=0, zipf_pct=0, third=tg.THIRD_UNIFORM)
    rng = np.random.default_rng(step0 % 1000 + int(old_frac * 100))
    h = hs.Handle(B, C, R, S, ratio, T)
    try:
        hs.hs_set_copy_mode(h.h, mode)
        hs.hs_set_policy(h.h, policy)
        pool = h.host_pool()
        for b in range(B):
            pool[b, :C] = tg.rows(wl, 0, b, 0, C)
        states = [_random_state(rng, C, S, C - T, step0, old_frac) for _ in range(B)]
        hs.hs_import_state(h.h, np.stack([s[0] for s in states]), np.stack([s[1] for s in states]),
                           np.stack([s[2] for s in states]), step0)
        orc = []
        for b in range(B):
            o = oracle.RequestState(C, S, T, R, policy=policy)
            o.tok_slot[:], o.slot_tok[:], o.stamp[:] = states[b]
            orc.append(o)
        imported = np.stack([s[1] for s in states])
        steps = 4
        for s in range(steps):
            rows = np.stack([_rows(rng, orc[b].tok_slot, C - T, C, K, hit_frac=0.4 + 0.1 * s)
                             for b in range(B)])
            if s == 2:
                rows[1, ::3] = -1  # some padding
            dev_rows = torch.from_numpy(rows).cuda()
            out = torch.empty_like(dev_rows)
            hs.hs_resolve(h.h, dev_rows, K, out)
            out = out.cpu().numpy()
            for b in range(B):
                host = pool[b, :C]
                o_out, counts, err = orc[b].resolve(host, rows[b], step0 + s + 1)
                np.testing.assert_array_equal(out[b], o_out, err_msg="step %d request %d" % (s, b))
                assert err == 0
        tok, slot_tok, stamp, step = h.export_state()
        assert step == step0 + steps
        for b in range(B):
            np.testing.assert_array_equal(tok[b], orc[b].tok_slot)
            np.testing.assert_array_equal(slot_tok[b], orc[b].slot_tok)
            np.testing.assert_array_equal(stamp[b], orc[b].stamp)
            buf = h.export_buffer(b)
            refilled = np.nonzero(slot_tok[b] != imported[b])[0]
            assert len(refilled) > 0
            np.testing.assert_array_equal(buf[refilled], orc[b].buf[refilled])
    finally:
        h.close()


def test_import_rejects_unreachable_states():
    from hierarchical_kv_cache_hs_gb300 import hs
    B, C, S = 2, 64, 8
    h = hs.Handle(B, C, 16, S, 8, 0)
    try:
        tok = np.full((B, C), -1, np.int32)
        st = np.full((B, S), -1, np.int32)
        stamp = np.zeros((B, S), np.int32)
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 0) == 0
        st[0, 3] = 10
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == hs.HS_ERR_ARG  # not inverse
        tok[0, 10] = 3
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == 0
        stamp[1, 2] = 6
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == hs.HS_ERR_ARG  # stamp > step
        stamp[1, 2] = 5
        tok[1, 20] = 9
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == hs.HS_ERR_ARG  # slot out of range
        tok[1, 20] = -1
        st[1, 0] = C
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == hs.HS_ERR_ARG  # token out of range
        st[1, 0] = -1
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, -1) == hs.HS_ERR_ARG
        assert hs.hs_import_state_rc(h.h, tok, st, stamp, 5) == 0
        assert h.stats()["steps"] == 5
    finally:
        h.close()
