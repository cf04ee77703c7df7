"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

All work on this path is integer and byte work, so every comparison is exact
(bit-exact out_slot, tables, stamps, miss counts, counters and buffer bytes).
The five named workloads run at full size and full length; the edge cases
cover ragged sizes, the kernel limits, K = S, a single slot, a resident tail
that runs out, invalid and repeated indices, padding and empty steps, CUDA
graph replay and the host-buffer entry point.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from hierarchical_kv_cache_hs_gb300 import tracegen as tg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_all()
    import oracle
    oracle.build()


def _run_and_compare(wl, steps=None, requests=None, graph=False, trace=None, expect_err=0,
                     copy_mode=0, policy=0, cluster_size=0, seed=0):
    from gpu_harness import check_counters, compare, gpu_run
    res = gpu_run(wl, steps=steps, graph=graph, trace=trace, copy_mode=copy_mode, policy=policy,
                  cluster_size=cluster_size, seed=seed)
    try:
        tot, err = compare(wl, res, requests=requests)
        if requests is None:
            check_counters(wl, res, tot, err | expect_err)
        return res, tot
    finally:
        res.workload.close()


@pytest.mark.parametrize("name", ["tiny_b1_c8k", "b32_c32k_s4096"])
def test_parity_full(name):
    wl = tg.WORKLOADS[name]
    res, tot = _run_and_compare(wl)
    assert res.misses[0, 0].tolist() == [wl.K] * wl.B  # cold start: every index misses


def test_parity_b64_buffer_sweep():
    """Both buffer sizes of the 64-request, 64K-context workload, full length.

    HiSparse blog, "Efficient swap-in kernel": with LRU, 4096 slots miss far
    less than 2048.  Miss counts per step are reported by the bench."""
    per = {}
    for name in ("b64_c64k_s4096", "b64_c64k_s2048"):
        wl = tg.WORKLOADS[name]
        res, tot = _run_and_compare(wl)
        per[wl.S] = res.misses[0, 10:].sum()
    assert per[4096] < 0.9 * per[2048]


def test_parity_b256_growing_tail():
    wl = tg.WORKLOADS["b256_c32k_grow_tail512"]
    res, tot = _run_and_compare(wl)
    assert tot[2] > 0  # some tail tokens were resolved in place


def test_parity_b64_four_layers_tail4096():
    wl = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    _run_and_compare(wl)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_parity_layers_on_concurrent_streams(graph):
    """The four independent layers on one stream each (fork/join events)."""
    from gpu_harness import check_counters, compare, gpu_run
    wl = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    res = gpu_run(wl, steps=40, graph=graph, layer_streams=True)
    try:
        tot, err = compare(wl, res, requests=[0, 21, 63])
    finally:
        res.workload.close()


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_parity_layers_in_one_launch(graph):
    """The four layers' step as one grid (hs_resolve_layers)."""
    from gpu_harness import compare, gpu_run
    wl = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    res = gpu_run(wl, steps=40, graph=graph, one_launch=True)
    try:
        compare(wl, res, requests=[0, 21, 63])
    finally:
        res.workload.close()


def test_parity_uniform_misses_four_layers():
    """Misses spread uniformly over four 10 GB host pools, all layers in one
    launch; sampled requests of every layer against the oracle."""
    from gpu_harness import compare, gpu_run
    wl = tg.WORKLOADS["b64_c128k_l4_uniform"]
    res = gpu_run(wl, steps=24, one_launch=True)
    try:
        tot, err = compare(wl, res, requests=[0, 37, 63])
        assert tot[1] > 0 and err == 0
    finally:
        res.workload.close()


@pytest.mark.parametrize("row_bytes", [1152, 1040])
def test_parity_one_launch_mixed_layers(row_bytes):
    """One launch over layers that differ in policy, with a sliding tail fed by
    appends; every request of every layer against the oracle (both copy
    unrolls)."""
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = tg.Workload("layers_slide", 87, B=6, C=6144, K=384, S=768, T=256, host_ratio=8,
                     layers=3, steps=120, len0=3000, grow=1, carry_pct=60, zipf_pct=30,
                     third=tg.THIRD_RECENT, recent=1024, sliding=True, row_bytes=row_bytes)
    res = gpu_run(wl, one_launch=True, policy=[hs.HS_POLICY_LRU, hs.HS_POLICY_FIFO,
                                               hs.HS_POLICY_LRU])
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
        assert tot[1] > 0 and tot[2] > 0
    finally:
        res.workload.close()


def _random_workload(seed):
    """A small seeded workload with random sizes, tail (fixed or sliding),
    growth, layers and row size."""
    import random
    rng = random.Random(seed)
    S = rng.choice([1, 7, 64, 300, 1024, 2500])
    K = rng.randint(1, min(S, 900))
    T = rng.choice([0, 0, 16, 128])
    grow = T > 0 and rng.random() < 0.5
    sliding = grow and rng.random() < 0.5
    C = rng.randint(max(K, 8), 6000) + T
    ratio = -(-(C - T) // S)  # enough host rows for the cold tokens
    steps = rng.randint(5, 40)
    if sliding:
        # the tail holds the last T tokens written; the first row needs K tokens
        len0 = rng.randint(max(min(T, C - 8), K), C - 8)
        steps = min(steps, C - len0)
    else:
        len0 = C - T if grow else C  # a fixed tail starts empty when the context grows
    R = rng.choice([16, 1152, 1040, 4096])
    B = rng.choice([1, 3, 17, 40])
    carry = rng.choice([0, 50, 80])
    return tg.Workload("rand%d" % seed, 70 + seed, B=B, C=C, K=K, S=S, T=T, host_ratio=ratio,
                       layers=rng.choice([1, 1, 2, 3]), steps=steps, len0=len0,
                       grow=1 if grow else 0, carry_pct=carry, zipf_pct=rng.choice([0, 100 - carry - 10]),
                       third=rng.choice([tg.THIRD_ZIPF, tg.THIRD_UNIFORM]), row_bytes=R,
                       sliding=sliding)


def _wide_workload(seed):
    """Random sizes up to the kernel limits: S to 16384, K to 4096, rows to 64 KB."""
    import random
    rng = random.Random(seed)
    S = rng.choice([1, 2, 3, 5, 33, 127, 1000, 4095, 4096, 8191, 16384])
    K = rng.randint(1, min(S, 4096))
    if rng.random() < 0.2:
        K = min(S, 4096)
    T = rng.choice([0, 0, 1, 3, 64, 1000])
    grow = T > 0 and rng.random() < 0.5
    sliding = grow and rng.random() < 0.5
    R = 16 * rng.choice([1, 2, 3, 65, 72, 129, 256, 1024, 4096])
    B = rng.choice([1, 2, 16, 17, 64, 150])
    layers = rng.choice([1, 1, 2])
    C = rng.randint(max(K, 8), max(K, 8) + rng.choice([10, 1000, 30000])) + T
    # keep the pinned pools under ~3 GB and the device buffers under ~2 GB
    while layers * B * C * R > 3e9 or layers * B * (S + T) * R > 2e9:
        if B > 1:
            B = max(1, B // 2)
        elif layers > 1:
            layers = 1
        else:
            R = 16
            break
    ratio = -(-(C - T) // S)
    steps = rng.randint(3, 25)
    if sliding and max(min(T, C - 8), K) > C - 8:
        sliding = False
    if sliding:
        len0 = rng.randint(max(min(T, C - 8), K), C - 8)
        steps = min(steps, C - len0)
    else:
        len0 = C - T if grow else C
    carry = rng.choice([0, 50, 90])
    return tg.Workload("wide%d" % seed, 40 + seed % 30, B=B, C=C, K=K, S=S, T=T, host_ratio=ratio,
                       layers=layers, steps=steps, len0=len0, grow=1 if grow else 0,
                       carry_pct=carry, zipf_pct=rng.choice([0, 100 - carry - 5]),
                       third=rng.choice([tg.THIRD_ZIPF, tg.THIRD_UNIFORM]), row_bytes=R, sliding=sliding)


@pytest.mark.parametrize("seed", range(24))
def test_parity_wide_random(seed):
    """Seeded random workloads drawn up to the kernel limits, every request of
    every layer against the oracle."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _wide_workload(seed)
    rng = random.Random(9000 + seed)
    mode = rng.choice([0, 1, 2])
    pol = [rng.choice([0, 1]) for _ in range(wl.layers)]
    one = wl.layers > 1 and rng.random() < 0.5
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    res = gpu_run(wl, copy_mode=mode, policy=pol, one_launch=one)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(12))
def test_parity_wide_random_cluster(seed):
    """The wide random workloads in cluster mode (several CTAs per request),
    with a random cluster size."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _wide_workload(500 + seed)
    rng = random.Random(9500 + seed)
    pol = [rng.choice([0, 1]) for _ in range(wl.layers)]
    n = rng.choice([0, 2, 3, 4, 8, 16])
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    res = gpu_run(wl, copy_mode=hs.HS_COPY_CLUSTER, policy=pol, cluster_size=n)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(12))
def test_parity_random_multi_position(seed):
    """Seeded random draft-position steps: P rows per request that repeat one
    another's tokens and carry padding, random sizes, launch mode and policy."""
    import random
    import oracle
    from hierarchical_kv_cache_hs_gb300 import hs
    rng = random.Random(500 + seed)
    P = rng.choice([2, 3, 4])
    Kp = rng.randint(1, 300)
    S = P * Kp + rng.choice([0, 1, 100, 1000])
    C = rng.randint(P * Kp + 1, 9000)
    R = rng.choice([16, 1152, 1040])
    B = rng.choice([1, 5, 20])
    steps = rng.randint(3, 25)
    ratio = -(-C // S)
    policy = rng.choice([0, 1])
    wl = tg.Workload("multi%d" % seed, 60 + seed, B=B, C=C, K=Kp, S=S, T=0, host_ratio=ratio,
                     layers=P, steps=steps, len0=C, grow=0, carry_pct=rng.choice([0, 60]),
                     zipf_pct=30, third=tg.THIRD_ZIPF, row_bytes=R)
    rows = [tg.topk_trace(wl, layer=p_) for p_ in range(P)]
    nrng = np.random.default_rng(seed)
    for p_ in range(1, P):  # later positions repeat tokens of the first
        take = nrng.random(rows[p_].shape) < 0.4
        pick = nrng.integers(0, Kp, size=rows[p_].shape)
        rows[p_] = np.where(take, np.take_along_axis(rows[0], pick, axis=2), rows[p_])
    trace = np.ascontiguousarray(np.concatenate(rows, axis=2))  # [steps][B][P*K]
    trace[nrng.random(trace.shape) < 0.03] = -1  # padding
    h = hs.Handle(B, C, R, S, ratio, 0)
    try:
        hs.hs_set_copy_mode(h.h, rng.choice([0, 1, 2]))
        if seed % 3 == 2:  # a third of the seeds in cluster mode
            hs.hs_set_copy_mode(h.h, hs.HS_COPY_CLUSTER)
        hs.hs_set_policy(h.h, policy)
        pool = h.host_pool()
        for b in range(B):
            pool[b, :C] = tg.rows(wl, 0, b, 0, C)
        dev = torch.from_numpy(trace).cuda()
        out = torch.empty_like(dev)
        for s in range(steps):
            hs.hs_resolve_multi(h.h, dev[s], P, Kp, out[s])
        torch.cuda.synchronize()
        out = out.cpu().numpy()
        tok, slot_tok, stamp, step = h.export_state()
        stats = h.stats()
        tot_m = 0
        for b in range(B):
            st = oracle.RequestState(C, S, 0, R, policy=policy)
            host = pool[b, :C].copy()
            for s in range(steps):
                o, c, e = st.resolve(host, trace[s, b], s + 1, alias=True)
                np.testing.assert_array_equal(out[s, b], o, err_msg="step %d request %d" % (s, b))
                assert e == 0
                tot_m += c[1]
            np.testing.assert_array_equal(tok[b], st.tok_slot)
            np.testing.assert_array_equal(slot_tok[b], st.slot_tok)
            np.testing.assert_array_equal(stamp[b], st.stamp)
            occ = np.nonzero(st.slot_tok >= 0)[0]
            np.testing.assert_array_equal(h.export_buffer(b)[occ], st.buf[occ])
        assert stats["misses"] == tot_m and stats["err_bits"] == 0 and step == steps
    finally:
        h.close()


@pytest.mark.parametrize("seed", range(64))
def test_parity_random_workloads(seed):
    """Seeded random sizes (slots, top-k, tail, growth, layers, row size,
    batch) in a random launch mode and policy, every request of every layer
    against the oracle."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _random_workload(seed)
    rng = random.Random(1000 + seed)
    mode = rng.choice([0, 1, 2])
    policies = [rng.choice([0, 1]) for _ in range(wl.layers)]
    one = wl.layers > 1 and rng.random() < 0.5
    # more appends than fixed tail slots: the extra appends are refused and flagged
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    res = gpu_run(wl, copy_mode=mode, policy=policies, one_launch=one)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(24))
def test_parity_random_workloads_random_eviction(seed):
    """The random workloads with random eviction on most layers (each layer its
    own seed), in a random launch mode, every request of every layer against
    the oracle."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _random_workload(2000 + seed)
    rng = random.Random(3000 + seed)
    mode = rng.choice([0, 1, 2, 3])
    policies = [rng.choice([2, 2, 2, 0, 1]) for _ in range(wl.layers)]
    one = wl.layers > 1 and mode != 3 and rng.random() < 0.5
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    res = gpu_run(wl, copy_mode=mode, policy=policies, one_launch=one, seed=rng.getrandbits(64))
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(32))
def test_parity_random_workloads_cluster(seed):
    """The random workloads in cluster mode with a random cluster size (0 is
    the handle's default), every request of every layer against the oracle."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _random_workload(600 + seed)
    rng = random.Random(1600 + seed)
    policies = [rng.choice([0, 1]) for _ in range(wl.layers)]
    n = rng.choice([0, 0, 2, 3, 4, 5, 8, 16])
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    res = gpu_run(wl, copy_mode=hs.HS_COPY_CLUSTER, policy=policies, cluster_size=n)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(24))
def test_parity_random_noisy_traces(seed):
    """The random workloads with input errors mixed into every row: padding,
    indices below -1 or past the current length, and repeats of an earlier
    entry.  Those entries get -1 and the same error bits as the oracle; the
    rest of the step is unaffected."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _random_workload(100 + seed)
    rng = random.Random(2000 + seed)
    trace = np.stack([tg.topk_trace(wl, layer=l) for l in range(wl.layers)])  # [L][steps][B][K]
    nrng = np.random.default_rng(seed)
    u = nrng.random(trace.shape)
    trace[u < 0.03] = -1
    trace[(u >= 0.03) & (u < 0.04)] = wl.C + 5                     # past any length
    trace[(u >= 0.04) & (u < 0.045)] = -3                          # below -1
    if wl.K > 1:  # repeats: copy an earlier entry of the same row
        rep = (u >= 0.045) & (u < 0.07)
        rep[..., 0] = False
        idx = np.nonzero(rep)
        trace[idx] = trace[idx[:-1] + (nrng.integers(0, idx[-1]),)] if len(idx[-1]) else trace[idx]
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    mode = rng.choice([0, 1, 2])
    policy = [rng.choice([0, 1]) for _ in range(wl.layers)]
    one = wl.layers > 1 and rng.random() < 0.5
    if seed >= 16:  # the same kind of traces in cluster mode
        mode, one = hs.HS_COPY_CLUSTER, False
    res = gpu_run(wl, trace=trace, copy_mode=mode, policy=policy, one_launch=one,
                  cluster_size=[0, 2, 4, 8][seed % 4] if seed >= 16 else 0)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err | expect)
        if ((trace >= wl.C) | (trace < -1)).any():
            assert err & hs.HS_E_RANGE
    finally:
        res.workload.close()


@pytest.mark.parametrize("seed", range(8))
def test_noalloc_random_matches_handle_path(seed):
    """hs_resolve_noalloc on caller-owned state against hs_resolve, on random
    fixed-context sizes (with or without a resident tail)."""
    import random
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    k = 0
    while True:  # the next random workload without growth, one layer
        wl = _random_workload(300 + seed * 50 + k)
        k += 1
        if not wl.grow and not wl.sliding:
            break
    wl = wl.with_(layers=1)
    ref = GpuWorkload(wl, record=True)
    try:
        h = ref.handles[0]
        dev = "cuda"
        B, C, S, T, R, K = wl.B, wl.C, wl.S, wl.T, wl.row_bytes, wl.K
        tok_slot = torch.full((B, C), -1, dtype=torch.int32, device=dev)
        slot_tok = torch.full((B, S), -1, dtype=torch.int32, device=dev)
        stamp = torch.zeros((B, S), dtype=torch.int32, device=dev)
        lengths = torch.full((B,), C, dtype=torch.int32, device=dev)
        buf = torch.zeros((B, S + T, R), dtype=torch.uint8, device=dev)
        control = torch.zeros(8, dtype=torch.int32, device=dev)
        out = torch.full((wl.steps, B, K), -7, dtype=torch.int32, device=dev)
        for b in range(T and B):
            buf[b, S:] = torch.from_numpy(h.export_buffer(b)[S:]).to(dev)
        stream = torch.cuda.current_stream()
        for s in range(wl.steps):
            ref.launch_step(s, stream)
            hs.hs_resolve_noalloc(B, C, R, S, wl.H, T, ref.topk[0, s], K, out[s], tok_slot, slot_tok,
                                  stamp, lengths, hs.hs_host_pool(h.h), buf, control, stream)
        torch.cuda.synchronize()
        assert torch.equal(out, ref.out[0])
        tok_ref, slot_ref, stamp_ref, step_ref = h.export_state()
        np.testing.assert_array_equal(tok_slot.cpu().numpy(), tok_ref)
        np.testing.assert_array_equal(slot_tok.cpu().numpy(), slot_ref)
        np.testing.assert_array_equal(stamp.cpu().numpy(), stamp_ref)
        assert int(control[0]) == step_ref == wl.steps
        for b in range(B):
            occ = np.nonzero(slot_ref[b] >= 0)[0]
            np.testing.assert_array_equal(buf[b].cpu().numpy()[occ], h.export_buffer(b)[occ])
    finally:
        ref.close()


@pytest.mark.parametrize("seed", list(range(12)) + [12, 15, 18, 21])
def test_parity_random_entry_points(seed):
    """Random workloads through the other entry points: the whole run replayed
    from one CUDA graph, the copy-engine variant, or host buffers (against the
    device path step by step)."""
    import random
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = _random_workload(400 + seed)
    rng = random.Random(3000 + seed)
    one = wl.layers > 1 and rng.random() < 0.5
    expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
    kind = seed % 3
    if kind < 2:
        mode = rng.choice([0, 1, 2])
        if kind == 0 and seed >= 12:
            mode, one = hs.HS_COPY_CLUSTER, False  # graph replay in cluster mode
        res = gpu_run(wl, graph=kind == 0, copy_engine=kind == 1, one_launch=one and kind == 0,
                      copy_mode=mode, cluster_size=[0, 2, 4, 8][seed % 4] if mode == 3 else 0)
        try:
            tot, err = compare(wl, res)
            check_counters(wl, res, tot, err | expect)
        finally:
            res.workload.close()
        return
    a = GpuWorkload(wl, record=True)
    b = GpuWorkload(wl, record=False, host_trace=True)
    try:
        out_host = torch.empty((wl.layers, wl.B, wl.K), dtype=torch.int32).pin_memory()
        for s in range(wl.steps):
            a.launch_step(s, one_launch=one)
            b.host_step(s, out_host, one_launch=one)
            torch.cuda.synchronize()
            assert torch.equal(a.out[:, s].cpu(), out_host), s
        for ha, hb in zip(a.handles, b.handles):
            for x, y in zip(ha.export_state(), hb.export_state()):
                np.testing.assert_array_equal(x, y)
            assert ha.stats()["misses"] == hb.stats()["misses"]
    finally:
        a.close()
        b.close()


def test_handles_driven_from_two_host_threads():
    """Two handles, each created and stepped from its own host thread on its
    own stream at the same time; both match the oracle."""
    import threading
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wls = [_random_workload(900), _random_workload(901)]
    results, errors = [None, None], []

    def run(i):
        try:
            results[i] = gpu_run(wls[i], copy_mode=i + 1)  # each run makes its own stream
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for wl, res in zip(wls, results):
        try:
            tot, err = compare(wl, res)
            expect = hs.HS_E_APPEND if (wl.grow and not wl.sliding and wl.steps > wl.T) else 0
            check_counters(wl, res, tot, err | expect)
        finally:
            res.workload.close()


def test_parity_two_thousand_steps():
    """A long run: slots that go unused for more than 1023 steps leave the
    exact-age bins, so the victim search takes its radix-select path in the
    ordinary flow of steps."""
    wl = tg.Workload("long_run", 79, B=3, C=20000, K=64, S=256, T=0, host_ratio=80, layers=1,
                     steps=2000, len0=20000, grow=0, carry_pct=80, zipf_pct=20,
                     third=tg.THIRD_ZIPF)
    _run_and_compare(wl)


def test_create_accepts_a_pool_that_covers_the_cold_tokens():
    """15 host rows per slot cannot hold 1024 cold tokens at 64 slots (the CPU
    test checks the refusal), but with 64 tokens resident 960 are enough."""
    from hierarchical_kv_cache_hs_gb300 import hs
    rc, h = hs.hs_create_rc(4, 1024, 1152, 64, 15, 64)
    assert rc == hs.HS_OK and h
    hs.hs_destroy(h)


def test_one_launch_at_the_layer_limit():
    """HS_MAX_LAYERS (16) handles in one launch, against the oracle."""
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = tg.Workload("layers16", 76, B=5, C=3000, K=200, S=400, T=64, host_ratio=8,
                     layers=hs.HS_MAX_LAYERS, steps=12, len0=3000, grow=0, carry_pct=60,
                     zipf_pct=30, third=tg.THIRD_ZIPF)
    res = gpu_run(wl, one_launch=True, policy=[l % 2 for l in range(wl.layers)])
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
    finally:
        res.workload.close()


def test_one_launch_argument_checks():
    from hierarchical_kv_cache_hs_gb300 import hs
    a = hs.Handle(4, 2048, 64, 256, 8)
    b = hs.Handle(4, 2048, 64, 256, 8)
    c = hs.Handle(4, 2048, 64, 512, 4)   # other S
    d = hs.Handle(2, 2048, 64, 256, 8)   # other B
    try:
        t = torch.arange(128, dtype=torch.int32, device="cuda").repeat(4, 1).contiguous()
        o = torch.empty_like(t)
        rc = hs.hs_resolve_layers_rc
        assert rc([a.h, a.h], [t, t], 128, [o, o]) == hs.HS_ERR_ARG
        assert rc([a.h, c.h], [t, t], 128, [o, o]) == hs.HS_ERR_ARG
        assert rc([a.h, d.h], [t, t], 128, [o, o]) == hs.HS_ERR_ARG
        assert rc([a.h, b.h], [t, None], 128, [o, o]) == hs.HS_ERR_ARG
        assert rc([a.h, b.h], [t, t], 257, [o, o]) == hs.HS_ERR_TOPK_GT_SLOTS
        assert rc([a.h, b.h], [t, t], 128, [o, o]) == hs.HS_OK
        torch.cuda.synchronize()
        assert a.stats()["misses"] == 4 * 128 and b.stats()["misses"] == 4 * 128
    finally:
        for h in (a, b, c, d):
            h.close()


EDGE = {
    # ragged: K and S not multiples of the CTA width, B odd
    "ragged": tg.Workload("ragged", 91, B=3, C=5000, K=1000, S=3000, T=0, host_ratio=2, layers=1,
                          steps=30, len0=5000, grow=0, carry_pct=70, zipf_pct=30,
                          third=tg.THIRD_ZIPF),
    # K = S with no carry-over: nearly every index misses, every slot is a victim
    "k_equals_s": tg.Workload("k_equals_s", 92, B=4, C=9000, K=2048, S=2048, T=0, host_ratio=5,
                              layers=1, steps=20, len0=9000, grow=0, carry_pct=0, zipf_pct=0,
                              third=tg.THIRD_UNIFORM),
    # the kernel limits: K = 4096, S = 16384
    "max_sizes": tg.Workload("max_sizes", 93, B=2, C=65536, K=4096, S=16384, T=0, host_ratio=4,
                             layers=1, steps=12, len0=65536, grow=0, carry_pct=70, zipf_pct=30,
                             third=tg.THIRD_ZIPF),
    # one slot, one index
    "single_slot": tg.Workload("single_slot", 94, B=5, C=10, K=1, S=1, T=0, host_ratio=10,
                               layers=1, steps=30, len0=10, grow=0, carry_pct=0, zipf_pct=0,
                               third=tg.THIRD_UNIFORM),
    # small rows, many requests
    "small_rows": tg.Workload("small_rows", 95, B=300, C=2048, K=64, S=128, T=0, host_ratio=16,
                              layers=1, steps=25, len0=2048, grow=0, carry_pct=50, zipf_pct=25,
                              third=tg.THIRD_UNIFORM, row_bytes=16),
    # rows of 65 16-byte chunks: the 8-deep copy unroll, row groups that end mid-warp;
    # fused (20 requests) and split (5 requests)
    "odd_rows_fused": tg.Workload("odd_rows_fused", 85, B=20, C=3000, K=300, S=600, T=0,
                                  host_ratio=5, layers=1, steps=30, len0=3000, grow=0, carry_pct=60,
                                  zipf_pct=30, third=tg.THIRD_ZIPF, row_bytes=1040),
    "odd_rows_split": tg.Workload("odd_rows_split", 84, B=5, C=3000, K=300, S=600, T=0,
                                  host_ratio=5, layers=1, steps=30, len0=3000, grow=0, carry_pct=60,
                                  zipf_pct=30, third=tg.THIRD_ZIPF, row_bytes=1040),
    # 2 KB rows with a resident tail
    "wide_rows_tail": tg.Workload("wide_rows_tail", 83, B=17, C=4096, K=256, S=512, T=64,
                                  host_ratio=8, layers=1, steps=25, len0=4096, grow=0, carry_pct=60,
                                  zipf_pct=30, third=tg.THIRD_ZIPF, row_bytes=2048),
    # an odd top-k: the shared word array after the two 16-bit arrays (FIFO's hit
    # bitmap) must stay aligned
    "odd_k": tg.Workload("odd_k", 78, B=17, C=4000, K=301, S=512, T=0, host_ratio=8, layers=1,
                         steps=25, len0=4000, grow=0, carry_pct=60, zipf_pct=30,
                         third=tg.THIRD_ZIPF),
    # the largest row (64 KB): one row per warp group, many chunks per lane, no early fetch
    "max_rows": tg.Workload("max_rows", 82, B=16, C=512, K=64, S=128, T=0, host_ratio=4,
                            layers=1, steps=10, len0=512, grow=0, carry_pct=50, zipf_pct=30,
                            third=tg.THIRD_ZIPF, row_bytes=65536),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_parity_edge_sizes(name):
    _run_and_compare(EDGE[name])


@pytest.mark.parametrize("name", sorted(EDGE))
def test_parity_edge_sizes_cluster(name):
    """The edge sizes with a cluster of CTAs per request (4, or the default)."""
    from hierarchical_kv_cache_hs_gb300 import hs
    _run_and_compare(EDGE[name], copy_mode=hs.HS_COPY_CLUSTER, cluster_size=4)
    if EDGE[name].B <= 32:
        _run_and_compare(EDGE[name], steps=min(EDGE[name].steps, 10), copy_mode=hs.HS_COPY_CLUSTER)


SLIDE = tg.Workload("slide_b16_c8k_tail256", 89, B=16, C=8192, K=512, S=1024, T=256,
                    host_ratio=8, layers=1, steps=600, len0=4096, grow=1, carry_pct=60,
                    zipf_pct=30, third=tg.THIRD_RECENT, recent=1024, sliding=True)


@pytest.mark.parametrize("mode,policy", [(0, 0), (2, 0), (1, 1), (3, 0), (3, 1)])
def test_parity_sliding_tail(mode, policy):
    """A sliding tail: tokens that leave it are written back to the host pool
    and later come back through the hot buffer as ordinary misses."""
    res, tot = _run_and_compare(SLIDE, copy_mode=mode, policy=policy)
    assert tot[2] > 0 and tot[1] > 0


def test_parity_sliding_tail_graph():
    _run_and_compare(SLIDE, steps=64, graph=True, requests=[0, 7, 15])


def test_parity_tail_overflow():
    """A growing context that outruns its 16-token tail: appends past the tail
    latch HS_E_APPEND, indices past the length latch HS_E_RANGE."""
    wl = tg.Workload("tail_overflow", 96, B=3, C=616, K=64, S=128, T=16, host_ratio=5, layers=1,
                     steps=24, len0=600, grow=1, carry_pct=50, zipf_pct=25, third=tg.THIRD_RECENT,
                     recent=64)
    from gpu_harness import compare, gpu_run
    res = gpu_run(wl)
    try:
        tot, err = compare(wl, res)
        assert res.stats[0]["err_bits"] == err | 4
        assert err & 1
    finally:
        res.workload.close()


def _corrupt(trace, C, seed):
    rng = np.random.default_rng(seed)
    tr = trace.copy()
    L, steps, B, K = tr.shape
    for s in range(steps):
        for b in range(B):
            kind = rng.integers(0, 6)
            j = rng.integers(0, K, size=4)
            if kind == 0:
                tr[0, s, b, j] = -1                      # padding
            elif kind == 1:
                tr[0, s, b, j[0]] = C + int(rng.integers(0, 5))  # past the length
            elif kind == 2:
                tr[0, s, b, j[0]] = -2 - int(rng.integers(0, 5))  # below -1
            elif kind == 3:
                tr[0, s, b, j[1]] = tr[0, s, b, j[0]]    # repeated index
            elif kind == 4:
                tr[0, s, b, :] = -1                      # an empty row
    tr[0, 3] = -1                                         # a step with no work at all
    return tr


def test_parity_invalid_and_padding():
    wl = tg.Workload("invalid", 97, B=4, C=3000, K=256, S=512, T=0, host_ratio=6, layers=1,
                     steps=12, len0=3000, grow=0, carry_pct=70, zipf_pct=30, third=tg.THIRD_ZIPF)
    base = tg.topk_trace(wl)[None]
    tr = _corrupt(base, wl.C, 5)
    res, tot = _run_and_compare(wl, trace=tr)
    assert res.stats[0]["err_bits"] == 3
    assert (res.out[0, 3] == -1).all() and (res.misses[0, 3] == 0).all()


@pytest.mark.parametrize("mode", [1, 2, 3], ids=["fused", "split", "cluster"])
def test_graph_replay_matches_oracle(mode):
    """The whole step sequence captured in one CUDA graph and replayed."""
    for name in ("tiny_b1_c8k", "b32_c32k_s4096"):
        wl = tg.WORKLOADS[name]
        _run_and_compare(wl, steps=40, graph=True, copy_mode=mode)
    wl = tg.WORKLOADS["b256_c32k_grow_tail512"]
    _run_and_compare(wl, steps=24, graph=True, requests=[0, 101, 255], copy_mode=mode)


@pytest.mark.parametrize("name,mode", [("tiny_b1_c8k", 1), ("b32_c32k_s4096", 2),
                                       ("b64_c64k_s4096", 2), ("ragged", 1),
                                       ("max_sizes", 1), ("single_slot", 1),
                                       ("tiny_b1_c8k", 2), ("b32_c32k_s4096", 1),
                                       ("b64_c64k_s4096", 1), ("b64_c64k_s2048", 1),
                                       ("b256_c32k_grow_tail512", 3)])
def test_parity_other_launch_mode(name, mode):
    """The launch modes the default does not pick for a workload: one CTA per
    request (fused) and the resolve + copy pair (split) up to 128 requests,
    where the default is a cluster per request, and a cluster per request at
    256 requests, where the default is fused."""
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    _run_and_compare(wl, copy_mode=mode)


@pytest.mark.parametrize("placement", ["base", "huge"])
@pytest.mark.parametrize("name,mode", [("ragged", 3), ("odd_k", 2), ("b32_c32k_s4096", 1),
                                       ("b32_c32k_s4096", 3)])
def test_parity_host_pool_placement(placement, name, mode):
    """Both host-pool placements give the oracle's results: cudaHostAlloc, and
    anonymous memory advised for huge pages and registered with
    cudaHostRegister (forced here for pools of any size).  With the default
    placement, only pools of at least HS_POOL_HUGE_MIN_BYTES take the second."""
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    want = hs.HS_POOL_PAGES_BASE if placement == "base" else hs.HS_POOL_PAGES_HUGE
    if want == hs.HS_POOL_PAGES_HUGE and hs.hs_huge_page_bytes() == 0:
        pytest.skip("the host offers no transparent huge pages")
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    seen = []
    hs.hs_set_host_pool_pages(want)
    try:
        res = gpu_run(wl, copy_mode=mode, setup=lambda w: seen.extend(
            hs.hs_host_pool_pages(h.h) for h in w.handles))
    finally:
        hs.hs_set_host_pool_pages(hs.HS_POOL_PAGES_AUTO)
    try:
        assert seen == [want] * wl.layers
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
    finally:
        res.workload.close()
    # the default placement keeps pools below the size floor in cudaHostAlloc memory
    h = hs.Handle(wl.B, wl.C, wl.row_bytes, wl.S, wl.host_ratio, wl.T)
    try:
        assert hs.hs_host_pool_bytes(h.h) < hs.HS_POOL_HUGE_MIN_BYTES
        assert hs.hs_host_pool_pages(h.h) == hs.HS_POOL_PAGES_BASE
    finally:
        h.close()


def test_parity_pool_past_the_huge_page_floor():
    """A pool of HS_POOL_HUGE_MIN_BYTES or more takes the huge-page placement by
    default (where the host offers huge pages), and its steps match the oracle:
    16 requests with a 933,888-token context, 17.2 GB of pool, the default
    launch (a cluster per request); the first and last requests are compared."""
    from gpu_harness import compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    S, ratio = 2048, 456
    wl = tg.Workload("pool_17g", 23, B=16, C=S * ratio, K=1024, S=S, T=0, host_ratio=ratio,
                     layers=1, steps=6, len0=S * ratio, grow=0, carry_pct=70, zipf_pct=20,
                     third=tg.THIRD_UNIFORM)
    assert wl.B * wl.H * wl.row_bytes >= hs.HS_POOL_HUGE_MIN_BYTES
    seen = []
    res = gpu_run(wl, setup=lambda w: seen.extend(hs.hs_host_pool_pages(h.h) for h in w.handles))
    try:
        want = hs.HS_POOL_PAGES_HUGE if hs.hs_huge_page_bytes() > 0 else hs.HS_POOL_PAGES_BASE
        assert seen == [want]
        assert hs.hs_launch_mode(res.workload.handles[0].h) == hs.HS_COPY_CLUSTER
        compare(wl, res, requests=[0, wl.B - 1])
    finally:
        res.workload.close()


@pytest.mark.parametrize("name,mode", [("b32_c32k_s4096", 0), ("b32_c32k_s4096", 2),
                                       ("tiny_b1_c8k", 0), ("b256_c32k_grow_tail512", 0),
                                       ("ragged", 1), ("odd_k", 1), ("odd_k", 2),
                                       ("b32_c32k_s4096", 3), ("odd_k", 3)])
def test_parity_fifo_policy(name, mode):
    """FIFO eviction (hits keep their fill stamp) against the oracle's FIFO."""
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    res, tot = _run_and_compare(wl, copy_mode=mode, policy=1)


@pytest.mark.parametrize("name,mode", [("b32_c32k_s4096", 0), ("b32_c32k_s4096", 1),
                                       ("b32_c32k_s4096", 2), ("tiny_b1_c8k", 0),
                                       ("b256_c32k_grow_tail512", 0), ("ragged", 3), ("odd_k", 1),
                                       ("odd_k", 2), ("odd_k", 3), ("single_slot", 0), ("k_equals_s", 3),
                                       ("max_sizes", 3), ("small_rows", 2)])
def test_parity_random_policy(name, mode):
    """Random eviction (keys from SplitMix64 of seed, step, request and slot)
    against the oracle's, in every launch mode."""
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    _run_and_compare(wl, copy_mode=mode, policy=2, seed=0x5EED0000ABCD + len(name))


def test_parity_random_policy_sliding_graph_layers():
    """Random eviction with a sliding tail, replayed from one CUDA graph, and
    in the several-layer launch (each layer its own seed)."""
    from gpu_harness import compare, gpu_run
    _run_and_compare(SLIDE, copy_mode=3, policy=2, seed=99)
    _run_and_compare(SLIDE, steps=48, graph=True, requests=[0, 7, 15], policy=2, seed=7)
    wl = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    res = gpu_run(wl, steps=24, one_launch=True, policy=[2, 0, 2, 1], seed=1 << 40)
    try:
        compare(wl, res, requests=[0, 33, 63])
    finally:
        res.workload.close()


def test_random_misses_more_than_lru():
    wl = tg.WORKLOADS["b32_c32k_s4096"]
    per = {}
    for policy in (0, 2):
        res, tot = _run_and_compare(wl, steps=40, policy=policy, seed=3)
        per[policy] = tot[1]
    assert per[0] < per[2]


@pytest.mark.parametrize("name,ctas", [("b32_c32k_s4096", 1), ("b32_c32k_s4096", 48),
                                       ("odd_k", 3), ("ragged", 7), ("b256_c32k_grow_tail512", 48)])
def test_parity_split_copy_grid(name, ctas):
    """The split mode's copy kernel on a small grid (hs_set_copy_ctas): each warp
    takes a longer run of the flattened miss list, with the same results."""
    from gpu_harness import check_counters, compare, gpu_run
    from hierarchical_kv_cache_hs_gb300 import hs
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    res = gpu_run(wl, copy_mode=hs.HS_COPY_SPLIT,
                  setup=lambda w: [hs.hs_set_copy_ctas(h.h, ctas) for h in w.handles])
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
    finally:
        res.workload.close()


def test_fifo_misses_more_than_lru():
    wl = tg.WORKLOADS["b32_c32k_s4096"]
    per = {}
    for policy in (0, 1):
        res, tot = _run_and_compare(wl, steps=40, policy=policy)
        per[policy] = tot[1]
    assert per[0] < per[1]


@pytest.mark.parametrize("name", ["b32_c32k_s4096", "b256_c32k_grow_tail512", "ragged"])
def test_parity_copy_engine_variant(name):
    """hs_resolve_ce (host gather + one copy-engine transfer) against the oracle."""
    from gpu_harness import check_counters, compare, gpu_run
    wl = tg.WORKLOADS.get(name) or EDGE[name]
    res = gpu_run(wl, steps=min(wl.steps, 40), copy_engine=True)
    try:
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
    finally:
        res.workload.close()


@pytest.mark.parametrize("policy", [0, 2], ids=["lru", "random"])
@pytest.mark.parametrize("mode", [1, 2, 3], ids=["fused", "split", "cluster"])
def test_parity_multi_position(mode, policy):
    """Two draft positions per step: the second row repeats about half of the
    first's tokens; repeats share their first occurrence's slot."""
    import oracle
    from hierarchical_kv_cache_hs_gb300 import hs
    P, Kp, B, C, S, R = 2, 512, 24, 16384, 2048, 1152
    wl = tg.Workload("multi", 88, B=B, C=C, K=Kp, S=S, T=0, host_ratio=8, layers=2, steps=40,
                     len0=C, grow=0, carry_pct=70, zipf_pct=30, third=tg.THIRD_ZIPF)
    t0 = tg.topk_trace(wl, layer=0)
    t1 = tg.topk_trace(wl, layer=1)
    rng = np.random.default_rng(3)
    take = rng.random(t1.shape) < 0.5
    pick = rng.integers(0, Kp, size=t1.shape)
    t1 = np.where(take, np.take_along_axis(t0, pick, axis=2), t1)
    trace = np.ascontiguousarray(np.concatenate([t0, t1], axis=2))  # [steps][B][P*K]
    h = hs.Handle(B, C, R, S, 8, 0)
    try:
        hs.hs_set_copy_mode(h.h, mode)
        hs.hs_set_policy(h.h, policy)
        hs.hs_set_eviction_seed(h.h, 41)
        pool = h.host_pool()
        for b in range(B):
            pool[b, :C] = tg.rows(wl, 0, b, 0, C)
        dev = torch.from_numpy(trace).cuda()
        out = torch.empty_like(dev)
        for s in range(wl.steps):
            hs.hs_resolve_multi(h.h, dev[s], P, Kp, out[s])
        torch.cuda.synchronize()
        out = out.cpu().numpy()
        tok, slot_tok, stamp, step = h.export_state()
        stats = h.stats()
        tot_m = 0
        for b in range(B):
            st = oracle.RequestState(C, S, 0, R, policy=policy, req=b, seed=41)
            host = pool[b, :C].copy()
            for s in range(wl.steps):
                o, c, e = st.resolve(host, trace[s, b], s + 1, alias=True)
                np.testing.assert_array_equal(out[s, b], o, err_msg="step %d request %d" % (s, b))
                assert e == 0
                tot_m += c[1]
            np.testing.assert_array_equal(tok[b], st.tok_slot)
            np.testing.assert_array_equal(slot_tok[b], st.slot_tok)
            np.testing.assert_array_equal(stamp[b], st.stamp)
            buf = h.export_buffer(b)
            occ = np.nonzero(st.slot_tok >= 0)[0]
            np.testing.assert_array_equal(buf[occ], st.buf[occ])
        assert stats["misses"] == tot_m and stats["err_bits"] == 0
        # repeats really occurred, across and within positions
        assert (out[:, :, Kp:][take] >= 0).all()
    finally:
        h.close()


@pytest.mark.parametrize("step0", [100, 1 << 21, -5, 0x7FFFFFF0])
def test_corrupt_caller_state_is_contained(step0):
    """Tables a caller owns (hs_resolve_noalloc) may be garbage: out-of-range
    page-table and slot entries and stamps beyond the step counter.  The step
    must stay inside its buffers, return slots in range and latch HS_E_STATE;
    the context stays usable afterwards."""
    from hierarchical_kv_cache_hs_gb300 import hs
    B, C, S, K, R, ratio = 4, 4096, 512, 256, 64, 8
    rng = np.random.default_rng(11)
    h = hs.Handle(B, C, R, S, ratio, 0)  # only for its pinned host pool
    try:
        dev = "cuda"
        tok = rng.integers(-1, S, size=(B, C)).astype(np.int32)
        bad = rng.random((B, C)) < 0.2
        tok[bad] = rng.integers(S, 4 * S, size=bad.sum())
        tok[rng.random((B, C)) < 0.05] = -7
        slot_tok = rng.integers(-1, C, size=(B, S)).astype(np.int32)
        slot_tok[rng.random((B, S)) < 0.2] = 10 * C
        stamp = rng.integers(-50, 1 << 22, size=(B, S)).astype(np.int32)
        t_tok = torch.from_numpy(tok).to(dev)
        t_slot = torch.from_numpy(slot_tok).to(dev)
        t_stamp = torch.from_numpy(stamp).to(dev)
        lengths = torch.full((B,), C, dtype=torch.int32, device=dev)
        buf = torch.zeros((B, S, R), dtype=torch.uint8, device=dev)
        control = torch.zeros(8, dtype=torch.int32, device=dev)
        control[0] = step0  # step counter, out of range in the last two cases
        out = torch.empty((B, K), dtype=torch.int32, device=dev)
        for s in range(3):
            rows = np.stack([rng.choice(C, K, replace=False) for _ in range(B)]).astype(np.int32)
            hs.hs_resolve_noalloc(B, C, R, S, h.H, 0, torch.from_numpy(rows).to(dev), K, out,
                                  t_tok, t_slot, t_stamp, lengths, hs.hs_host_pool(h.h), buf,
                                  control)
            torch.cuda.synchronize()
            o = out.cpu().numpy()
            assert ((o == -1) | ((o >= 0) & (o < S))).all()
        ctl = control.cpu().numpy()
        assert ctl[0] == step0 + 3 and ctl[1] & hs.HS_E_STATE
        # the context is still healthy
        h2 = hs.Handle(2, 1024, 32, 64, 16)
        try:
            row = torch.arange(64, dtype=torch.int32, device=dev).repeat(2, 1).contiguous()
            hs.hs_resolve(h2.h, row, 64, torch.empty_like(row))
            assert h2.stats()["misses"] == 128 and h2.stats()["err_bits"] == 0
        finally:
            h2.close()
    finally:
        h.close()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_layers_host_matches_device_path(pinned):
    """hs_resolve_layers_host (host top-k in, host out_slot back) against
    hs_resolve_layers on the same steps: identical slots and state."""
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    wl = tg.Workload("layers_host", 80, B=8, C=4096, K=256, S=512, T=128, host_ratio=8, layers=3,
                     steps=16, len0=4096, grow=0, carry_pct=60, zipf_pct=30, third=tg.THIRD_ZIPF)
    a = GpuWorkload(wl, record=True)
    b = GpuWorkload(wl, record=False)
    try:
        stream = torch.cuda.current_stream()
        trace = a.topk.cpu()
        if pinned:
            trace = trace.pin_memory()
        out = torch.empty((wl.layers, wl.B, wl.K), dtype=torch.int32)
        if pinned:
            out = out.pin_memory()
        L = wl.layers
        for s in range(wl.steps):
            a.launch_step(s, stream, one_launch=True)
            hs.hs_resolve_layers_host([h.h for h in b.handles], [trace[l, s] for l in range(L)], wl.K,
                                      [out[l] for l in range(L)], stream)
            torch.cuda.synchronize()
            assert torch.equal(out, a.out[:, s].cpu()), s
        for ha, hb in zip(a.handles, b.handles):
            for x, y in zip(ha.export_state(), hb.export_state()):
                np.testing.assert_array_equal(x, y)
    finally:
        a.close()
        b.close()


def test_layers_host_refuses_before_staging():
    """hs_resolve_layers_host with pageable host buffers makes every check of
    hs_resolve_layers before it stages anything: a second handle with fewer
    slots (whose staging buffers are smaller than the first handle's K), one
    with another batch size, a handle given twice and a K beyond the slots
    each return an error; no handle's state or counters change, the output
    buffers stay untouched, and the following steps still match the oracle."""
    from gpu_harness import GpuResult, check_counters, compare
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    wl = tg.Workload("layers_host_checks", 81, B=4, C=4096, K=400, S=512, T=0, host_ratio=8,
                     layers=2, steps=8, len0=4096, grow=0, carry_pct=60, zipf_pct=30,
                     third=tg.THIRD_ZIPF)
    w = GpuWorkload(wl, record=True)
    small = hs.Handle(wl.B, wl.C, wl.row_bytes, 256, 16)   # S = 256 < K
    other_b = hs.Handle(2, wl.C, wl.row_bytes, wl.S, 8)
    try:
        stream = torch.cuda.current_stream()
        L = wl.layers
        misses = np.zeros((L, wl.steps, wl.B), dtype=np.int32)
        for s in range(3):
            w.launch_step(s, stream, one_launch=True)
            for layer, h in enumerate(w.handles):
                hs.hs_stats(h.h, misses[layer, s])
        trace = w.topk.cpu().numpy()            # pageable host memory
        out = np.full((L, wl.B, wl.K), -7, dtype=np.int32)
        before = [(h.export_state(), h.stats()) for h in w.handles + [small]]
        h0, h1 = w.handles[0].h, w.handles[1].h
        rc = hs.lib.hs_resolve_layers_host
        P = hs._ptr_array

        def call(handles, K=wl.K):
            return rc(P(handles), len(handles), P([trace[0, 3]] * len(handles)), K,
                      P([out[0]] * len(handles)), None)

        assert call([h0, small.h]) == hs.HS_ERR_ARG
        assert call([small.h, h0]) == hs.HS_ERR_ARG
        assert call([small.h]) == hs.HS_ERR_TOPK_GT_SLOTS
        assert call([h0, other_b.h]) == hs.HS_ERR_ARG
        assert call([h0, h1, h0]) == hs.HS_ERR_ARG
        assert call([h0, h1], K=wl.S + 1) == hs.HS_ERR_TOPK_GT_SLOTS
        torch.cuda.synchronize()
        assert (out == -7).all()
        after = [(h.export_state(), h.stats()) for h in w.handles + [small]]
        for (sa, ca), (sb, cb) in zip(before, after):
            for x, y in zip(sa, sb):
                np.testing.assert_array_equal(x, y)
            assert ca == cb
        for s in range(3, wl.steps):
            w.launch_step(s, stream, one_launch=True)
            for layer, h in enumerate(w.handles):
                hs.hs_stats(h.h, misses[layer, s])
        torch.cuda.synchronize()
        res = GpuResult()
        res.misses = misses
        res.out = w.out.cpu().numpy()
        res.trace = w.topk.cpu().numpy()
        res.stats = [h.stats() for h in w.handles]
        res.state = [h.export_state() for h in w.handles]
        res.workload = w
        res.policy = 0
        tot, err = compare(wl, res)
        check_counters(wl, res, tot, err)
    finally:
        small.close()
        other_b.close()
        w.close()


def test_reset_requests_admits_new_requests():
    """Continuous batching: after 12 steps, batch slots 1 and 4 take new
    requests (slot 4 with a shorter length) and the run goes on.  Those
    requests must match a fresh oracle state started at step 13; the others
    must not notice.  An id outside the batch latches HS_E_RANGE only."""
    import oracle
    from gpu_harness import oracle_request
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    wl = tg.Workload("admit", 81, B=6, C=5000, K=300, S=600, T=0, host_ratio=9, layers=1,
                     steps=24, len0=5000, grow=0, carry_pct=60, zipf_pct=30, third=tg.THIRD_ZIPF)
    w = GpuWorkload(wl, record=True)
    try:
        h = w.handles[0]
        stream = torch.cuda.current_stream()
        ids = torch.tensor([1, 4], dtype=torch.int32, device="cuda")
        lens = torch.tensor([wl.C, wl.C - 100], dtype=torch.int32, device="cuda")
        for s in range(wl.steps):
            if s == 12:
                hs.hs_reset_requests(h.h, ids, 2, lens, stream)
            w.launch_step(s, stream)
        torch.cuda.synchronize()
        out = w.out.cpu().numpy()[0]
        trace = w.topk.cpu().numpy()[0]
        tok, slot_tok, stamp, step = h.export_state()
        assert step == wl.steps
        err = 0
        for b in range(wl.B):
            host = tg.rows(wl, 0, b, 0, wl.cold)
            if b in (1, 4):
                st1, o1, _, e1 = oracle.run_request(wl.C, wl.S, wl.T, wl.row_bytes, host, trace[:12, b])
                length = wl.C if b == 1 else wl.C - 100
                st, o2, _, e2 = oracle.run_request(wl.C, wl.S, wl.T, wl.row_bytes, host, trace[12:, b],
                                                   length=length, step0=12)
                outs = np.concatenate([o1, o2])
                err |= int(np.bitwise_or.reduce(np.concatenate([e1, e2])))
            else:
                st, outs, _, e = oracle.run_request(wl.C, wl.S, wl.T, wl.row_bytes, host, trace[:, b])
                err |= int(np.bitwise_or.reduce(e))
            np.testing.assert_array_equal(out[:, b], outs, err_msg="request %d" % b)
            np.testing.assert_array_equal(tok[b], st.tok_slot)
            np.testing.assert_array_equal(slot_tok[b], st.slot_tok)
            np.testing.assert_array_equal(stamp[b], st.stamp)
            buf = h.export_buffer(b)
            occ = np.nonzero(st.slot_tok >= 0)[0]
            np.testing.assert_array_equal(buf[occ], st.buf[occ])
        assert h.stats()["err_bits"] == err
        # an id outside the batch: nothing changes but the error bit
        bad = torch.tensor([wl.B + 3], dtype=torch.int32, device="cuda")
        hs.hs_reset_requests(h.h, bad, 1, None, stream)
        torch.cuda.synchronize()
        tok2, slot_tok2, stamp2, _ = h.export_state()
        assert (tok2 == tok).all() and (slot_tok2 == slot_tok).all() and (stamp2 == stamp).all()
        assert h.stats()["err_bits"] & hs.HS_E_RANGE
    finally:
        w.close()


def test_resolve_host_matches_device_path():
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload
    wl = tg.WORKLOADS["b32_c32k_s4096"]
    steps = 16
    a = GpuWorkload(wl, steps=steps, record=True, host_trace=True)
    b = GpuWorkload(wl, steps=steps, record=False, host_trace=True)
    try:
        out_host = torch.empty((1, wl.B, wl.K), dtype=torch.int32).pin_memory()
        for s in range(steps):
            a.launch_step(s)
            b.host_step(s, out_host)
            torch.cuda.synchronize()
            assert torch.equal(a.out[0, s].cpu(), out_host[0])
        ta, tb = a.handles[0].export_state(), b.handles[0].export_state()
        for x, y in zip(ta[:3], tb[:3]):
            np.testing.assert_array_equal(x, y)
        assert hs.hs_stats(a.handles[0].h) == hs.hs_stats(b.handles[0].h)
        # pageable (unmapped) host buffers take the staged path
        c = GpuWorkload(wl, steps=steps, record=False)
        try:
            pageable_in = c.topk.cpu().numpy()
            pageable_out = np.empty((wl.B, wl.K), dtype=np.int32)
            for s in range(steps):
                hs.hs_resolve_host(c.handles[0].h, np.ascontiguousarray(pageable_in[0, s]), wl.K,
                                   pageable_out)
                assert (a.out[0, s].cpu().numpy() == pageable_out).all()
        finally:
            c.close()
    finally:
        a.close()
        b.close()


def test_device_errors_leave_context_usable():
    """K > S and oversized K are refused on the host; the handle still works."""
    from hierarchical_kv_cache_hs_gb300 import hs
    h = hs.Handle(2, 1024, 32, 64, 16)
    try:
        topk = torch.zeros((2, 128), dtype=torch.int32, device="cuda")
        out = torch.empty_like(topk)
        assert hs.hs_resolve_rc(h.h, topk, 128, out) == hs.HS_ERR_TOPK_GT_SLOTS
        assert hs.hs_resolve_rc(h.h, topk, 0, out) == hs.HS_ERR_ARG
        row = torch.arange(64, dtype=torch.int32, device="cuda").repeat(2, 1).contiguous()
        out = torch.empty_like(row)
        hs.hs_resolve(h.h, row, 64, out)
        st = h.stats()
        assert st["misses"] == 128 and st["steps"] == 1 and st["err_bits"] == 0
    finally:
        h.close()


def test_cluster_size_settings():
    """hs_set_cluster_size: 0 picks the default (16 or 8 CTAs up to 4
    requests, 5 beyond), 2..HS_MAX_CLUSTER are taken when the device runs
    them, other values are refused; cluster mode is one launch per step."""
    from hierarchical_kv_cache_hs_gb300 import hs
    h = hs.Handle(4, 8192, 1152, 1024, 8)
    try:
        auto = hs.hs_cluster_size(h.h)
        assert auto in (8, 16)  # up to 4 requests: wide clusters
        assert hs.hs_launch_mode(h.h) == hs.HS_COPY_CLUSTER  # the default takes them
        with pytest.raises(hs.HsError):
            hs.hs_set_cluster_size(h.h, 1)
        with pytest.raises(hs.HsError):
            hs.hs_set_cluster_size(h.h, -1)
        with pytest.raises(hs.HsError):
            hs.hs_set_cluster_size(h.h, hs.HS_MAX_CLUSTER + 1)
        for n in (2, 3, 8):
            hs.hs_set_cluster_size(h.h, n)
            assert hs.hs_cluster_size(h.h) == n
        hs.hs_set_cluster_size(h.h, 0)
        assert hs.hs_cluster_size(h.h) == auto
        hs.hs_set_copy_mode(h.h, hs.HS_COPY_CLUSTER)
        assert hs.hs_resolve_launches(h.h) == 1
    finally:
        h.close()
    big = hs.Handle(200, 4096, 64, 256, 16)
    try:
        assert hs.hs_cluster_size(big.h) == 5  # the size cluster mode would take
        # beyond HS_CLUSTER_MAX_BATCH requests the default takes one CTA per request
        assert hs.hs_launch_mode(big.h) == hs.HS_COPY_FUSED
        hs.hs_set_copy_mode(big.h, hs.HS_COPY_CLUSTER)
        assert hs.hs_launch_mode(big.h) == hs.HS_COPY_CLUSTER
    finally:
        big.close()
