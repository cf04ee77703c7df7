"""Run a synthetic swap-in workload through the C ABI.

Sets up one handle per layer, fills each pinned host pool with the seeded KV
rows, writes the resident tail (fixed context) or uploads the per-step rows
to append (growing context), and uploads the top-k trace to the device.
Every resolve goes through ``hs_resolve`` / ``hs_append``; this file only
prepares inputs and issues calls.  torch provides device memory and streams.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import hs
from . import tracegen as tg


class GpuWorkload:
    """Handles, inputs and output buffers of one workload on one GPU.

    ``steps`` decode steps of trace are generated (default: the workload's).
    With ``record=True`` every step's out_slot is kept on the device
    ([layers][steps][B][K]); otherwise one [layers][B][K] buffer is reused.
    """

    def __init__(self, wl: tg.Workload, steps: Optional[int] = None, record: bool = False,
                 device: str = "cuda", threads: Optional[int] = None, host_trace: bool = False,
                 request_offset: int = 0, copy_mode: int = hs.HS_COPY_AUTO):
        self.wl = wl
        self.steps = wl.steps if steps is None else int(steps)
        self.device = torch.device(device)
        self.record = record
        self.layers = wl.layers
        B, K, R = wl.B, wl.K, wl.row_bytes
        reqs = list(range(request_offset, request_offset + B))
        self.handles = []
        for layer in range(wl.layers):
            h = hs.Handle(B, wl.C, R, wl.S, wl.host_ratio, wl.T)
            self.handles.append(h)
            hs.hs_set_copy_mode(h.h, copy_mode)
            # Cold rows of request b live at pool row t of request slot b.
            self._fill_pool(h, layer, reqs, threads)
            if wl.sliding:
                # The tail holds the last T tokens written.
                hs.hs_set_tail_mode(h.h, hs.HS_TAIL_SLIDING)
                hs.hs_set_lengths(h.h, np.full(B, wl.len0, dtype=np.int32))
                first = max(wl.len0 - wl.T, 0)
                for i, b in enumerate(reqs):
                    hs.hs_set_tail_rows(h.h, i, first, tg.rows(wl, layer, b, first, wl.len0 - first))
            elif wl.grow:
                hs.hs_set_lengths(h.h, np.full(B, wl.len0, dtype=np.int32))
            elif wl.T > 0:
                for i, b in enumerate(reqs):
                    rows = tg.rows(wl, layer, b, wl.cold, wl.T)
                    hs.hs_set_tail_rows(h.h, i, wl.cold, rows)
        # Top-k trace: [layers][steps][B][K] int32.
        host = np.empty((wl.layers, self.steps, B, K), dtype=np.int32)
        for layer in range(wl.layers):
            tg.topk_trace(wl, layer=layer, steps=self.steps, requests=reqs, threads=threads,
                          out=host[layer])
        self.topk = torch.from_numpy(host).to(self.device)
        self.topk_host = torch.from_numpy(host).pin_memory() if host_trace else None
        # Rows appended before each step (growing context): [layers][steps][B][R].
        self.append_rows = None
        if wl.grow:
            ap = np.empty((wl.layers, self.steps, B, R), dtype=np.uint8)
            for layer in range(wl.layers):
                for i, b in enumerate(reqs):
                    ap[layer, :, i, :] = tg.rows(wl, layer, b, wl.len0, self.steps)
            self.append_rows = torch.from_numpy(ap).to(self.device)
        if record:
            self.out = torch.full((wl.layers, self.steps, B, K), -7, dtype=torch.int32,
                                  device=self.device)
        else:
            self.out = torch.full((wl.layers, B, K), -7, dtype=torch.int32, device=self.device)
        self.requests = reqs
        # The uploads and fills above ran on the current stream; steps may be
        # launched on any other, so they must be complete first.
        torch.cuda.synchronize(self.device)

    def _fill_pool(self, h, layer, reqs, threads):
        wl = self.wl
        base = hs.hs_host_pool(h.h)
        R, H = wl.row_bytes, wl.H
        # The generator keys rows by the request id; the pool is indexed by position.
        from concurrent.futures import ThreadPoolExecutor
        jobs = [(i, b, t0, min(4096, wl.cold - t0))
                for i, b in enumerate(reqs) for t0 in range(0, wl.cold, 4096)]

        def one(job):
            i, b, t0, n = job
            tg.fill_rows_ptr(wl, layer, b, t0, n, base + (i * H + t0) * R, R)

        with ThreadPoolExecutor(tg._workers(threads)) as ex:
            list(ex.map(one, jobs))
        self._touch_pool(h)

    def _touch_pool(self, h):
        """Read the whole pool once from the GPU (hs_h2d_read into a scratch
        buffer).  The GPU's first accesses to freshly pinned host pages pay an
        address-translation warm-up (measured on the 4-layer, 38 GB workload:
        its first steps took 0.65-1.23 ms instead of 0.54 ms); a serving pool
        lives for hours, so steps are measured on a warm one."""
        base, n = hs.hs_host_pool(h.h), hs.hs_host_pool_bytes(h.h)
        chunk = 1 << 28
        scratch = torch.empty(min(chunk, max(n, 16)), dtype=torch.uint8, device=self.device)
        off = 0
        while off + 16 <= n:
            k = min(chunk, n - off) // 16 * 16
            hs.hs_h2d_read(base + off, scratch.data_ptr(), k)
            off += k
        torch.cuda.synchronize()
        del scratch

    def out_at(self, layer: int, step: int) -> torch.Tensor:
        return self.out[layer, step] if self.record else self.out[layer]

    def launch_step(self, s: int, stream=None, copy_engine: bool = False,
                    layer_streams=None, one_launch: bool = False) -> int:
        """Enqueue step s for every layer; returns the number of kernel launches.

        ``copy_engine`` uses the copy-engine comparison variant (hs_resolve_ce),
        which synchronises the stream inside every call.  ``layer_streams``
        (one torch stream per layer) runs the independent layers concurrently:
        each waits for ``stream`` at the start and ``stream`` waits for all of
        them at the end, so one layer's resolve overlaps another's row fetch.
        ``one_launch`` resolves all layers in one launch (hs_resolve_layers)."""
        wl = self.wl
        if one_launch:
            n = 0
            if self.append_rows is not None:
                for layer, h in enumerate(self.handles):
                    hs.hs_append(h.h, self.append_rows[layer, s], stream)
                    n += 1
            L = len(self.handles)
            hs.hs_resolve_layers([h.h for h in self.handles], [self.topk[l, s] for l in range(L)],
                                 wl.K, [self.out_at(l, s) for l in range(L)], stream)
            return n + 1
        if layer_streams is not None:
            main = stream if stream is not None else torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(main)
            n = 0
            for layer, h in enumerate(self.handles):
                ls = layer_streams[layer]
                ls.wait_event(fork)
                if self.append_rows is not None:
                    hs.hs_append(h.h, self.append_rows[layer, s], ls)
                    n += 1
                hs.hs_resolve(h.h, self.topk[layer, s], wl.K, self.out_at(layer, s), ls)
                n += hs.hs_resolve_launches(h.h)
                join = torch.cuda.Event()
                join.record(ls)
                main.wait_event(join)
            return n
        n = 0
        for layer, h in enumerate(self.handles):
            if self.append_rows is not None:
                hs.hs_append(h.h, self.append_rows[layer, s], stream)
                n += 1
            if copy_engine:
                hs.hs_resolve_ce(h.h, self.topk[layer, s], wl.K, self.out_at(layer, s), stream)
                n += 2
            else:
                hs.hs_resolve(h.h, self.topk[layer, s], wl.K, self.out_at(layer, s), stream)
                n += hs.hs_resolve_launches(h.h)
        return n

    def host_step(self, s: int, out_host: torch.Tensor, stream=None, one_launch: bool = False) -> None:
        """Step s from host buffers (hs_resolve_host, or hs_resolve_layers_host
        with ``one_launch``), for end-to-end timing.

        The top-k rows and results are passed as raw addresses into the pinned
        [layers][steps][B][K] trace and the [layers][B][K] output."""
        wl = self.wl
        row = wl.B * wl.K * 4
        base_in = self.topk_host.data_ptr()
        base_out = out_host.data_ptr()
        if one_launch:
            if self.append_rows is not None:
                for layer, h in enumerate(self.handles):
                    hs.hs_append(h.h, self.append_rows[layer, s], stream)
            L = len(self.handles)
            hs.hs_resolve_layers_host([h.h for h in self.handles],
                                      [base_in + (layer * self.steps + s) * row for layer in range(L)],
                                      wl.K, [base_out + layer * row for layer in range(L)], stream)
            return
        for layer, h in enumerate(self.handles):
            if self.append_rows is not None:
                hs.hs_append(h.h, self.append_rows[layer, s], stream)
            hs.hs_resolve_host(h.h, base_in + (layer * self.steps + s) * row, wl.K,
                               base_out + layer * row, stream)

    def reset(self) -> None:
        """Back to the start state (a sliding tail's written-back host rows stay)."""
        wl = self.wl
        for layer, h in enumerate(self.handles):
            hs.hs_reset(h.h)
            if wl.grow or wl.sliding:
                hs.hs_set_lengths(h.h, np.full(wl.B, wl.len0, dtype=np.int32))
            if wl.sliding:
                first = max(wl.len0 - wl.T, 0)
                for i, b in enumerate(self.requests):
                    hs.hs_set_tail_rows(h.h, i, first, tg.rows(wl, layer, b, first, wl.len0 - first))

    def close(self) -> None:
        for h in self.handles:
            h.close()
        self.handles = []
