"""Run a workload on the GPU through the C ABI and compare it, request by
request, with the CPU oracle.  Used by the GPU parity tests and the smoke check.

Every comparison is exact (integer and byte work): per-step out_slot, per-step
miss counts, the final token->slot / slot->token tables and stamps, the step
counter, the cumulative counters, and the bytes of every occupied buffer slot
and every written tail slot.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from hierarchical_kv_cache_hs_gb300 import hs
from hierarchical_kv_cache_hs_gb300 import tracegen as tg
from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload


class GpuResult:
    pass


def set_cluster_size(h, n):
    """Cluster-mode CTAs per request; a size the device cannot run falls back to 8."""
    try:
        hs.hs_set_cluster_size(h, n)
    except hs.HsError as e:
        if e.code != hs.HS_ERR_LIMIT or n <= 8:
            raise
        hs.hs_set_cluster_size(h, 8)


def gpu_run(wl, steps=None, trace=None, graph=False, setup=None, copy_mode=hs.HS_COPY_AUTO,
            policy=hs.HS_POLICY_LRU, copy_engine=False, layer_streams=False, one_launch=False,
            cluster_size=0, seed=0):
    """Run ``steps`` steps; ``trace`` [layers][steps][B][K] replaces the generated one.

    ``policy`` is one eviction policy for every layer, or a list with one per layer;
    ``seed`` is random eviction's seed (layer l's handle takes seed + l).
    ``cluster_size``: CTAs per request in cluster mode (0 = the handle's default)."""
    w = GpuWorkload(wl, steps=steps, record=True, copy_mode=copy_mode)
    if cluster_size:
        for h in w.handles:
            set_cluster_size(h.h, cluster_size)
    for layer, h in enumerate(w.handles):
        hs.hs_set_policy(h.h, policy[layer] if isinstance(policy, (list, tuple)) else policy)
        hs.hs_set_eviction_seed(h.h, seed + layer)
    res_policy = policy
    if setup is not None:
        setup(w)
    if trace is not None:
        w.topk = torch.from_numpy(np.ascontiguousarray(trace, dtype=np.int32)).cuda()
    steps = w.steps
    res = GpuResult()
    res.misses = np.zeros((wl.layers, steps, wl.B), dtype=np.int32)
    stream = torch.cuda.Stream()
    # inputs set up above (a replaced trace, the policies) are on the current
    # stream: the steps' stream starts after them
    stream.wait_stream(torch.cuda.current_stream())
    lstreams = [torch.cuda.Stream() for _ in range(wl.layers)] if layer_streams else None
    if graph:
        # Warm the kernels up outside the capture, then restart from the empty state.
        with torch.cuda.stream(stream):
            w.launch_step(0, stream)
        stream.synchronize()
        w.reset()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(steps):
                w.launch_step(s, torch.cuda.current_stream(), layer_streams=lstreams,
                              one_launch=one_launch)
        g.replay()
        torch.cuda.synchronize()
        res.misses = None  # per-step counts are not observable inside one graph
    else:
        with torch.cuda.stream(stream):
            for s in range(steps):
                w.launch_step(s, stream, copy_engine=copy_engine, layer_streams=lstreams,
                              one_launch=one_launch)
                for layer, h in enumerate(w.handles):
                    hs.hs_stats(h.h, res.misses[layer, s])
    torch.cuda.synchronize()
    res.out = w.out.cpu().numpy()
    res.trace = w.topk.cpu().numpy()
    res.stats = [h.stats() for h in w.handles]
    res.state = [h.export_state() for h in w.handles]
    res.workload = w
    res.policy = res_policy
    res.seed = seed
    return res


def oracle_request(wl, layer, b, trace_lb, steps, policy=0, seed=0):
    host = tg.rows(wl, layer, b, 0, wl.cold)
    append_rows = tg.rows(wl, layer, b, wl.len0, steps) if wl.grow else None
    tail_init = None
    if wl.T > 0 and (wl.sliding or not wl.grow):
        first = max(wl.len0 - wl.T, 0) if wl.sliding else wl.cold
        last = wl.len0 if wl.sliding else wl.C
        tail = tg.rows(wl, layer, b, first, last - first)

        def tail_init(st, tail=tail, first=first):
            for i in range(tail.shape[0]):
                t = first + i
                st.buf[wl.S + t % wl.T] = tail[i]
    length = wl.len0 if (wl.grow or wl.sliding) else wl.C
    st, outs, counts, errs = oracle.run_request(
        wl.C, wl.S, wl.T, wl.row_bytes, host, trace_lb, length=length, append_rows=append_rows,
        tail_init=tail_init, policy=policy, sliding=wl.sliding, req=b, seed=seed)
    st.host_rows = host
    return st, outs, counts, errs


def compare(wl, res, requests=None, layers=None):
    """Compare the GPU run with the oracle on the given requests; returns oracle totals."""
    steps = res.out.shape[1]
    layers = range(wl.layers) if layers is None else layers
    requests = range(wl.B) if requests is None else requests
    jobs = [(l, b) for l in layers for b in requests]
    R = wl.row_bytes

    def one(job):
        layer, b = job
        policy = getattr(res, "policy", 0)
        if isinstance(policy, (list, tuple)):
            policy = policy[layer]
        st, outs, counts, errs = oracle_request(wl, layer, b, res.trace[layer, :, b], steps,
                                                policy=policy, seed=getattr(res, "seed", 0) + layer)
        tok, slot_tok, stamp, step = res.state[layer]
        ctx = "layer %d request %d" % (layer, b)
        np.testing.assert_array_equal(res.out[layer, :, b], outs, err_msg=ctx + " out_slot")
        if res.misses is not None:
            np.testing.assert_array_equal(res.misses[layer, :, b], counts[:, 1], err_msg=ctx + " misses")
        np.testing.assert_array_equal(tok[b], st.tok_slot, err_msg=ctx + " tok_slot")
        np.testing.assert_array_equal(slot_tok[b], st.slot_tok, err_msg=ctx + " slot_tok")
        np.testing.assert_array_equal(stamp[b], st.stamp, err_msg=ctx + " stamp")
        assert step == steps
        buf = res.workload.handles[layer].export_buffer(b)
        occ = np.nonzero(st.slot_tok >= 0)[0]
        np.testing.assert_array_equal(buf[occ], st.buf[occ], err_msg=ctx + " buffer bytes")
        if wl.T > 0:
            last = int(st.len[0])
            first = max(last - wl.T, 0) if wl.sliding else wl.cold
            toks = np.arange(first, last)
            tslots = wl.S + toks % wl.T
            np.testing.assert_array_equal(buf[tslots], st.buf[tslots], err_msg=ctx + " tail bytes")
        if wl.sliding:
            # rows written back to the host pool by the appends
            pool = res.workload.handles[layer].host_pool()[b]
            lo, hi = max(wl.len0 - wl.T, 0), max(int(st.len[0]) - wl.T, 0)
            np.testing.assert_array_equal(pool[lo:hi], st.host_rows[lo:hi],
                                          err_msg=ctx + " written-back host rows")
        return counts.sum(axis=0), int(np.bitwise_or.reduce(errs)) if len(errs) else 0

    results = oracle.parallel_map(one, jobs)
    tot = np.zeros(3, dtype=np.int64)
    err = 0
    res.layer_err = {}
    for (layer, _), (c, e) in zip(jobs, results):
        tot += c
        err |= e
        res.layer_err[layer] = res.layer_err.get(layer, 0) | e
    return tot, err


def check_counters(wl, res, tot, err):
    """Cumulative counters must equal the oracle's sums (all requests compared).

    Each layer's handle latches its own error bits: they must equal its
    layer's oracle bits, plus the bits of ``err`` that the oracle replay does
    not model (a refused append), which every handle is expected to carry."""
    hits = sum(s["hits"] for s in res.stats)
    misses = sum(s["misses"] for s in res.stats)
    inplace = sum(s["inplace"] for s in res.stats)
    assert (hits, misses, inplace) == tuple(int(x) for x in tot)
    assert sum(s["bytes_copied"] for s in res.stats) == misses * wl.row_bytes
    layer_err = getattr(res, "layer_err", None) or {}
    oracle_err = 0
    for e in layer_err.values():
        oracle_err |= e
    extra = err & ~oracle_err  # bits passed in by the caller, not from the replay
    for layer, s in enumerate(res.stats):
        expect = (layer_err[layer] | extra) if layer in layer_err else err
        assert s["err_bits"] == expect, (layer, s["err_bits"], expect)
