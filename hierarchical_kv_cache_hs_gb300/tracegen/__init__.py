"""Seeded synthetic inputs for the HiSparse swap-in path.

The swap-in kernel of the HiSparse blog ("Efficient swap-in kernel" section)
consumes, every decode step, the DSA indexer's top-k token indices
(top_k = 2048 in the blog's launch configurations) and KV rows that live in a
pinned host pool.  No indexer, model or dataset is available here, so these
inputs are synthetic: per-step top-k rows mixing carry-over from the previous
step, Zipf(1.1)-distributed positions and a uniform or recent-window component,
plus uniform random KV row bytes (576 bf16 = 1152 bytes per token).

This module holds none of the method's arithmetic.  It is the one piece of
code shared by the CUDA path's callers and the CPU oracle.  The generator
itself is C (``tracegen.c``); this file compiles it, describes the workloads
and runs the generator over requests in threads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Iterable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tracegen.c")
_LIB_PATH = os.path.join(_HERE, "libtracegen.so")

THIRD_ZIPF = 0
THIRD_UNIFORM = 1
THIRD_RECENT = 2


def build(force: bool = False) -> str:
    """Compile ``libtracegen.so`` next to its source (plain gcc, portable C)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("workload", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("len0", ctypes.c_int32),
        ("grow", ctypes.c_int32),
        ("carry_pct", ctypes.c_int32),
        ("zipf_pct", ctypes.c_int32),
        ("third", ctypes.c_int32),
        ("recent", ctypes.c_int32),
        ("zipf_a", ctypes.c_double),
    ]


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.tg_zipf_cdf.argtypes = [ctypes.c_double, ctypes.c_int32, ctypes.c_void_p]
        lib.tg_zipf_cdf.restype = ctypes.c_int
        lib.tg_trace_request.argtypes = [ctypes.POINTER(_Params), ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_int64]
        lib.tg_trace_request.restype = ctypes.c_int
        lib.tg_fill_rows.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_int64]
        lib.tg_fill_rows.restype = ctypes.c_int
        lib.tg_stream_value.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.tg_stream_value.restype = ctypes.c_uint64
        lib.tg_splitmix64.argtypes = [ctypes.c_uint64]
        lib.tg_splitmix64.restype = ctypes.c_uint64
        lib.tg_len_at.argtypes = [ctypes.POINTER(_Params), ctypes.c_int32]
        lib.tg_len_at.restype = ctypes.c_int32
        _lib_handle = lib
    return _lib_handle


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes of the swap-in state plus the trace recipe.

    B requests, context capacity C tokens, K indices per top-k row, S hot-buffer
    slots per request, T resident-tail tokens (0 = no mixed residency),
    host pool of host_ratio * S rows per request, ``layers`` independent
    layers, ``steps`` decode steps.  The top-k row of step s is drawn over the
    current length len0 + grow * (s + 1).
    """
    name: str
    wid: int
    B: int
    C: int
    K: int
    S: int
    T: int
    host_ratio: int
    layers: int
    steps: int
    len0: int
    grow: int
    carry_pct: int
    zipf_pct: int
    third: int
    recent: int = 0
    zipf_a: float = 1.1
    row_bytes: int = 1152
    seed: int = 0
    sliding: bool = False   # the tail holds the last T tokens written (else [C - T, C))

    @property
    def H(self) -> int:
        return self.host_ratio * self.S

    @property
    def cold(self) -> int:
        """Number of host-backed token positions, C - T."""
        return self.C - self.T

    def len_at(self, step: int) -> int:
        return self.len0 + self.grow * (step + 1)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the swap-in benchmark plan.  Names state what they are.
WORKLOADS = {
    # 1 request, 8K context, top-k 256 into 512 slots, 70 % carry-over + Zipf.
    "tiny_b1_c8k": Workload("tiny_b1_c8k", 1, B=1, C=8192, K=256, S=512, T=0, host_ratio=16,
                            layers=1, steps=64, len0=8192, grow=0, carry_pct=70, zipf_pct=30,
                            third=THIRD_ZIPF),
    # 32 requests, 32K context, 4096 slots, 70 / 20 / 10 carry / Zipf / uniform.
    "b32_c32k_s4096": Workload("b32_c32k_s4096", 2, B=32, C=32768, K=2048, S=4096, T=0,
                               host_ratio=8, layers=1, steps=200, len0=32768, grow=0,
                               carry_pct=70, zipf_pct=20, third=THIRD_UNIFORM),
    # 64 requests, 64K context, buffer sweep 4096 vs 2048 slots on one trace.
    "b64_c64k_s4096": Workload("b64_c64k_s4096", 3, B=64, C=65536, K=2048, S=4096, T=0,
                               host_ratio=16, layers=1, steps=200, len0=65536, grow=0,
                               carry_pct=70, zipf_pct=30, third=THIRD_ZIPF),
    "b64_c64k_s2048": Workload("b64_c64k_s2048", 3, B=64, C=65536, K=2048, S=2048, T=0,
                               host_ratio=32, layers=1, steps=200, len0=65536, grow=0,
                               carry_pct=70, zipf_pct=30, third=THIRD_ZIPF),
    # 256 requests, context 32768 growing one token per step into a 512-token
    # resident device tail; 60 / 30 / 10 carry / Zipf / last-4096 window.
    "b256_c32k_grow_tail512": Workload("b256_c32k_grow_tail512", 4, B=256, C=32768 + 512, K=2048,
                                       S=4096, T=512, host_ratio=8, layers=1, steps=512,
                                       len0=32768, grow=1, carry_pct=60, zipf_pct=30,
                                       third=THIRD_RECENT, recent=4096),
    # 64 requests, 128K context, 4 independent layers, 6144 slots, last 4096
    # tokens resident on the device and resolved in place.
    "b64_c128k_l4_tail4096": Workload("b64_c128k_l4_tail4096", 5, B=64, C=131072, K=2048, S=6144,
                                      T=4096, host_ratio=21, layers=4, steps=256, len0=131072,
                                      grow=0, carry_pct=70, zipf_pct=30, third=THIRD_ZIPF),
    # Stress case beyond the five: the 4-layer shape without a tail, the 30 % of
    # each row that is not carried over drawn uniformly over the whole context,
    # so misses land anywhere in four 10 GB host pools.
    "b64_c128k_l4_uniform": Workload("b64_c128k_l4_uniform", 5, B=64, C=131072, K=2048, S=6144,
                                     T=0, host_ratio=22, layers=4, steps=256, len0=131072,
                                     grow=0, carry_pct=70, zipf_pct=0, third=THIRD_UNIFORM),
}


def _params(wl: Workload) -> _Params:
    return _Params(wl.seed, wl.wid, wl.K, wl.len0, wl.grow, wl.carry_pct, wl.zipf_pct,
                   wl.third, wl.recent, wl.zipf_a)


_cdf_cache = {}


def zipf_cdf(a: float, n: int) -> np.ndarray:
    """Cumulative Zipf weights sum_{p<=i} (p+1)^-a for i < n (float64)."""
    key = (float(a), int(n))
    if key not in _cdf_cache:
        arr = np.empty(n, dtype=np.float64)
        rc = _lib().tg_zipf_cdf(float(a), int(n), arr.ctypes.data)
        if rc != 0:
            raise ValueError("bad Zipf table size %d" % n)
        _cdf_cache[key] = arr
    return _cdf_cache[key]


def _workers(threads: Optional[int]) -> int:
    if threads is not None:
        return max(1, int(threads))
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def topk_trace(wl: Workload, layer: int = 0, steps: Optional[int] = None,
               requests: Optional[Sequence[int]] = None, threads: Optional[int] = None,
               out: Optional[np.ndarray] = None) -> np.ndarray:
    """Top-k rows of ``steps`` steps for the given requests: int32 [steps][len(requests)][K]."""
    steps = wl.steps if steps is None else int(steps)
    reqs = list(range(wl.B)) if requests is None else [int(r) for r in requests]
    nmax = wl.len_at(steps - 1)
    cdf = zipf_cdf(wl.zipf_a, nmax)
    if out is None:
        out = np.empty((steps, len(reqs), wl.K), dtype=np.int32)
    assert out.shape == (steps, len(reqs), wl.K) and out.dtype == np.int32 and out.flags.c_contiguous
    prm = _params(wl)
    lib = _lib()
    stride = len(reqs) * wl.K
    base = out.ctypes.data

    def one(i):
        rc = lib.tg_trace_request(ctypes.byref(prm), cdf.ctypes.data, int(nmax), int(layer),
                                  int(reqs[i]), int(steps), base + 4 * i * wl.K, int(stride))
        if rc != 0:
            raise RuntimeError("trace generation failed for request %d" % reqs[i])

    with ThreadPoolExecutor(_workers(threads)) as ex:
        list(ex.map(one, range(len(reqs))))
    return out


def fill_rows_ptr(wl: Workload, layer: int, b: int, t0: int, n: int, dst_ptr: int,
                  dst_stride: Optional[int] = None) -> None:
    """Write the bytes of tokens [t0, t0+n) of (layer, b) to a raw host pointer."""
    stride = wl.row_bytes if dst_stride is None else int(dst_stride)
    rc = _lib().tg_fill_rows(wl.seed, wl.wid, int(layer), int(b), int(t0), int(n),
                             wl.row_bytes, int(dst_ptr), stride)
    if rc != 0:
        raise RuntimeError("row generation failed")


def rows(wl: Workload, layer: int, b: int, t0: int, n: int) -> np.ndarray:
    """Bytes of tokens [t0, t0+n) of (layer, b): uint8 [n][row_bytes]."""
    arr = np.empty((n, wl.row_bytes), dtype=np.uint8)
    if n:
        fill_rows_ptr(wl, layer, b, t0, n, arr.ctypes.data)
    return arr


def fill_host_pool(wl: Workload, layer: int, pool_ptr: int, requests: Iterable[int] = None,
                   threads: Optional[int] = None, chunk: int = 4096) -> None:
    """Fill a [B][H][R] host pool at ``pool_ptr`` with the cold rows [0, C-T) of every request."""
    reqs = list(range(wl.B)) if requests is None else list(requests)
    R, H = wl.row_bytes, wl.H
    jobs = []
    for b in reqs:
        for t0 in range(0, wl.cold, chunk):
            jobs.append((b, t0, min(chunk, wl.cold - t0)))

    def one(job):
        b, t0, n = job
        fill_rows_ptr(wl, layer, b, t0, n, pool_ptr + ((b * H + t0) * R), R)

    with ThreadPoolExecutor(_workers(threads)) as ex:
        list(ex.map(one, jobs))


def splitmix64(x: int) -> int:
    return int(_lib().tg_splitmix64(x & 0xFFFFFFFFFFFFFFFF))


def stream_value(key: int, ctr: int) -> int:
    return int(_lib().tg_stream_value(key & 0xFFFFFFFFFFFFFFFF, ctr & 0xFFFFFFFFFFFFFFFF))
