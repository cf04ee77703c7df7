"""hs_resolve_noalloc against hs_resolve.

hs_resolve_noalloc serves callers that cannot let a library allocate device
memory -- for instance an engine that has reserved nearly all of HBM for its
own KV pool, or a decode loop where an allocation would stall the device.
They own every piece of state and pass it in; the library keeps the per-step
miss lists in a fixed device array instead of allocating them.

Here the test (standing in for such a caller) allocates the state with torch,
shares the read-only pinned host pool of an ordinary handle, and runs two
steps in a row through both entry points on the same top-k rows.  The buffer
has as many slots as a row has indices, so the second step evicts: its
misses take LRU victims and write the evicted tokens out of the page table.
Results must be identical: out_slot, both tables, stamps, the buffer bytes of
every occupied slot, the step counter and the miss counter.

This file is collected last so that a failure here does not hide the others.
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


@pytest.mark.parametrize("resident_tail", [0, 256])
def test_noalloc_matches_handle_path(resident_tail):
    from hierarchical_kv_cache_hs_gb300 import hs
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    from hierarchical_kv_cache_hs_gb300.workload import GpuWorkload

    wl = tg.Workload("noalloc_check", 98, B=8, C=16384 + resident_tail, K=1024, S=1024,
                     T=resident_tail, host_ratio=16, layers=1, steps=2, len0=16384 + resident_tail,
                     grow=0, carry_pct=70, zipf_pct=30, third=tg.THIRD_ZIPF)
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
        control = torch.zeros(8, dtype=torch.int32, device=dev)  # one hs_control_t (32 bytes)
        out = torch.full((2, B, K), -7, dtype=torch.int32, device=dev)
        if T:
            # the resident tail rows, as the handle got them at set-up
            for b in range(B):
                buf[b, S:] = torch.from_numpy(h.export_buffer(b)[S:]).to(dev)
        pool = hs.hs_host_pool(h.h)
        stream = torch.cuda.current_stream()
        per_step = np.zeros((2, B), dtype=np.int32)
        for s in range(2):
            ref.launch_step(s, stream)
            hs.hs_resolve_noalloc(B, C, R, S, wl.H, T, ref.topk[0, s], K, out[s], tok_slot,
                                  slot_tok, stamp, lengths, pool, buf, control, stream)
            torch.cuda.synchronize()
            stats = h.stats(per_step[s])

        # every request missed more rows than it has slots: the second step evicted
        assert (per_step.sum(axis=0) > S).all()
        assert torch.equal(out, ref.out[0])
        tok_ref, slot_ref, stamp_ref, step_ref = h.export_state()
        np.testing.assert_array_equal(tok_slot.cpu().numpy(), tok_ref)
        np.testing.assert_array_equal(slot_tok.cpu().numpy(), slot_ref)
        np.testing.assert_array_equal(stamp.cpu().numpy(), stamp_ref)
        ctl = control.cpu().numpy()
        assert ctl[0] == step_ref == 2
        assert ctl[1] == stats["err_bits"] == 0
        assert int(ctl[4:6].view(np.uint64)[0]) == stats["misses"] > 0
        for b in range(B):
            mine = buf[b].cpu().numpy()
            theirs = h.export_buffer(b)
            occ = np.nonzero(slot_ref[b] >= 0)[0]
            np.testing.assert_array_equal(mine[occ], theirs[occ])
            if T:
                np.testing.assert_array_equal(mine[S:], theirs[S:])
        if T:
            assert stats["inplace"] == int(ctl[6:8].view(np.uint64)[0])
    finally:
        ref.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from hierarchical_kv_cache_hs_gb300 import hs
    rc = hs.lib.hs_resolve_noalloc(300, 4096, 1152, 4096, 4096, 0, 1, 2048, 1, 1, 1, 1, 1, 1, 1, 1, None)
    assert rc == hs.HS_ERR_LIMIT  # 300 * 2048 > HS_NOALLOC_MAX_ENTRIES
    rc = hs.lib.hs_resolve_noalloc(4, 4096, 1152, 1024, 4096, 0, 1, 2048, 1, 1, 1, 1, 1, 1, 1, 1, None)
    assert rc == hs.HS_ERR_TOPK_GT_SLOTS


def _state(B, C, S, T, R, dev="cuda"):
    return dict(tok_slot=torch.full((B, C), -1, dtype=torch.int32, device=dev),
                slot_tok=torch.full((B, S), -1, dtype=torch.int32, device=dev),
                stamp=torch.zeros((B, S), dtype=torch.int32, device=dev),
                lengths=torch.full((B,), C, dtype=torch.int32, device=dev),
                buf=torch.zeros((B, S + T, R), dtype=torch.uint8, device=dev),
                control=torch.zeros(8, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("placement", ["base", "huge"])
def test_noalloc_refuses_misaligned_pointers_and_short_pools(placement):
    """Host-side checks before anything is enqueued: a pool that the driver
    reports shorter than B * host_rows * R bytes, and pointers that break the
    kernels' alignment, return HS_ERR_ARG and leave the caller's state as it
    was; a correct call afterwards still runs.  The pool is a handle's, in
    either placement: cudaHostAlloc, or a cudaHostRegister registration of
    exactly the pool's bytes."""
    from hierarchical_kv_cache_hs_gb300 import hs
    want = hs.HS_POOL_PAGES_BASE if placement == "base" else hs.HS_POOL_PAGES_HUGE
    if want == hs.HS_POOL_PAGES_HUGE and hs.hs_huge_page_bytes() == 0:
        pytest.skip("the host offers no transparent huge pages")
    # a 4 MiB pool (2 requests x 2048 rows x 1 KiB), a whole number of pages
    B, C, S, K, R, ratio = 2, 1024, 128, 64, 1024, 16
    hs.hs_set_host_pool_pages(want)
    try:
        h = hs.Handle(B, C, R, S, ratio, 0)  # only for its pinned host pool
    finally:
        hs.hs_set_host_pool_pages(hs.HS_POOL_PAGES_AUTO)
    try:
        assert hs.hs_host_pool_pages(h.h) == want
        st = _state(B, C, S, 0, R)
        topk = torch.arange(K, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
        out = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
        pool = hs.hs_host_pool(h.h)

        def call(host_rows=h.H, pool=pool, buf=st["buf"].data_ptr(), control=st["control"].data_ptr(),
                 stamp=st["stamp"].data_ptr()):
            return hs.lib.hs_resolve_noalloc(B, C, R, S, host_rows, 0, topk.data_ptr(), K,
                                             out.data_ptr(), st["tok_slot"].data_ptr(),
                                             st["slot_tok"].data_ptr(), stamp,
                                             st["lengths"].data_ptr(), pool, buf, control, None)

        # the pool allocation holds B * H rows; twice as many would run past it
        assert call(host_rows=2 * h.H) == hs.HS_ERR_ARG
        assert call(pool=pool + 16, host_rows=h.H) == hs.HS_ERR_ARG  # 16 bytes short at the end
        assert call(buf=st["buf"].data_ptr() + 4) == hs.HS_ERR_ARG
        assert call(pool=pool + 8, host_rows=h.H - 1) == hs.HS_ERR_ARG
        assert call(control=st["control"].data_ptr() + 4) == hs.HS_ERR_ARG
        assert call(stamp=st["stamp"].data_ptr() + 2) == hs.HS_ERR_ARG
        torch.cuda.synchronize()
        assert int(st["control"].abs().sum()) == 0 and bool((out == -7).all())
        assert bool((st["tok_slot"] == -1).all()) and bool((st["slot_tok"] == -1).all())
        # a pool that starts one row in and stops one row short of the end is inside it
        assert call(pool=pool + R, host_rows=h.H - 1) == hs.HS_OK
        torch.cuda.synchronize()
        assert int(st["control"][0]) == 1 and bool((out >= 0).all())
    finally:
        h.close()


def test_noalloc_first_call_inside_a_capture_is_refused():
    """In a fresh process, a first call made while its stream is being captured
    returns HS_ERR_ARG and enqueues nothing; the next call, outside the
    capture, does the set-up and runs."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = r'''
import sys
sys.path.insert(0, %r)
import torch
from hierarchical_kv_cache_hs_gb300 import hs
B, C, S, K, R = 2, 1024, 128, 64, 64
h = hs.Handle(B, C, R, S, 8, 0)
tok = torch.full((B, C), -1, dtype=torch.int32, device="cuda")
slot = torch.full((B, S), -1, dtype=torch.int32, device="cuda")
stamp = torch.zeros((B, S), dtype=torch.int32, device="cuda")
lens = torch.full((B,), C, dtype=torch.int32, device="cuda")
buf = torch.zeros((B, S, R), dtype=torch.uint8, device="cuda")
ctl = torch.zeros(8, dtype=torch.int32, device="cuda")
topk = torch.arange(K, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous()
out = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
def call(stream):
    return hs.lib.hs_resolve_noalloc(B, C, R, S, h.H, 0, topk.data_ptr(), K, out.data_ptr(),
                                     tok.data_ptr(), slot.data_ptr(), stamp.data_ptr(),
                                     lens.data_ptr(), hs.hs_host_pool(h.h), buf.data_ptr(),
                                     ctl.data_ptr(), stream)
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
torch.cuda.synchronize()
with torch.cuda.graph(g, stream=s):
    rc = call(s.cuda_stream)
assert rc == hs.HS_ERR_ARG, rc
torch.cuda.synchronize()
assert int(ctl[0]) == 0 and bool((out == -7).all())
assert call(None) == hs.HS_OK
torch.cuda.synchronize()
assert int(ctl[0]) == 1 and bool((out >= 0).all())
h.close()
print("capture check ok")
''' % root
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "capture check ok" in r.stdout, r.stdout + r.stderr
