"""hs_resolve_noalloc against hs_resolve.

hs_resolve_noalloc serves callers that cannot let a library allocate device
memory -- for instance an engine that has reserved nearly all of HBM for its
own KV pool, or a decode loop where an allocation would stall the device.
They own every piece of state and pass it in; the library keeps the per-step
miss lists in a fixed device array instead of allocating them.

Here the test (standing in for such a caller) allocates the state with torch,
shares the read-only pinned host pool of an ordinary handle, and runs two
steps in a row through both entry points on the same top-k rows.  Results
must be identical: out_slot, both tables, stamps, the buffer bytes of every
occupied slot, the step counter and the miss counter.

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

    wl = tg.Workload("noalloc_check", 98, B=8, C=16384 + resident_tail, K=1024, S=2048,
                     T=resident_tail, host_ratio=8, layers=1, steps=2, len0=16384 + resident_tail,
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
        for s in range(2):
            ref.launch_step(s, stream)
            hs.hs_resolve_noalloc(B, C, R, S, wl.H, T, ref.topk[0, s], K, out[s], tok_slot,
                                  slot_tok, stamp, lengths, pool, buf, control, stream)
        torch.cuda.synchronize()

        assert torch.equal(out, ref.out[0])
        tok_ref, slot_ref, stamp_ref, step_ref = h.export_state()
        np.testing.assert_array_equal(tok_slot.cpu().numpy(), tok_ref)
        np.testing.assert_array_equal(slot_tok.cpu().numpy(), slot_ref)
        np.testing.assert_array_equal(stamp.cpu().numpy(), stamp_ref)
        ctl = control.cpu().numpy()
        stats = h.stats()
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
