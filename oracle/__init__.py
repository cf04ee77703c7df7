"""CPU oracle of the HiSparse swap-in path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``hs_oracle.c`` (plain sequential C, one request at a
time; every step cites the passage it follows).  This file compiles it and
drives it over steps and requests.  Requests are independent, so whole
workloads run one request per thread (ctypes releases the GIL).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

E_RANGE = 1
E_DUP = 2
E_NOROOM = 8

POLICY_LRU = 0
POLICY_FIFO = 1
POLICY_RANDOM = 2


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, no CUDA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
                    _SRC, "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib_handle = None


def load_library(path: str):
    """Load a compiled oracle (the default one, or a test's planted-mistake copy)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.or_init.argtypes = [i32, i32, P, P, P]
    lib.or_init.restype = None
    lib.or_resolve.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, i32, P, P]
    lib.or_resolve.restype = i32
    if hasattr(lib, "or_resolve_policy"):
        lib.or_resolve_policy.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, i32, P, P,
                                          i32]
        lib.or_resolve_policy.restype = i32
    if hasattr(lib, "or_resolve_ex"):
        lib.or_resolve_ex.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, i32, P, P,
                                      i32, i32]
        lib.or_resolve_ex.restype = i32
        lib.or_append_sliding.argtypes = [i32, i32, i32, i32, P, P, P, P]
        lib.or_append_sliding.restype = i32
    if hasattr(lib, "or_resolve_full"):
        lib.or_resolve_full.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, i32, P, P,
                                        i32, i32, i32]
        lib.or_resolve_full.restype = i32
    if hasattr(lib, "or_resolve_keyed"):
        lib.or_resolve_keyed.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, i32, P, P,
                                         i32, i32, i32, i32, ctypes.c_uint64]
        lib.or_resolve_keyed.restype = i32
        lib.or_splitmix64_at.argtypes = [ctypes.c_uint64]
        lib.or_splitmix64_at.restype = ctypes.c_uint64
    lib.or_append.argtypes = [i32, i32, i32, i32, P, P, P]
    lib.or_append.restype = i32
    return lib


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        _lib_handle = load_library(_LIB_PATH)
    return _lib_handle


class RequestState:
    """State of one request: tables, stamps, device-buffer model and length."""

    def __init__(self, C: int, S: int, T: int, R: int, length: Optional[int] = None, lib=None,
                 policy: int = POLICY_LRU, sliding: bool = False, req: int = 0, seed: int = 0):
        self.lib = lib if lib is not None else _lib()
        self.policy = int(policy)
        # random eviction keys on the request's index and the seed
        self.req, self.seed = int(req), int(seed) & ((1 << 64) - 1)
        self.sliding = bool(sliding)
        self.C, self.S, self.T, self.R = int(C), int(S), int(T), int(R)
        self.tok_slot = np.empty(C, dtype=np.int32)
        self.slot_tok = np.empty(S, dtype=np.int32)
        self.stamp = np.empty(S, dtype=np.int32)
        self.buf = np.zeros((S + T, R), dtype=np.uint8)
        self.len = np.array([C if length is None else length], dtype=np.int32)
        self.lib.or_init(self.C, self.S, self.tok_slot.ctypes.data, self.slot_tok.ctypes.data,
                       self.stamp.ctypes.data)

    def resolve(self, host: np.ndarray, topk: np.ndarray, step: int, alias: bool = False):
        """Resolve one top-k row at ``step``; host is uint8 [C-T][R] by token.

        ``alias``: the row is several positions' rows concatenated, and a
        repeated token takes its first occurrence's slot instead of being an
        error.  Returns (out int32 [K], (hits, misses, inplace), err_bits).
        """
        topk = np.ascontiguousarray(topk, dtype=np.int32)
        assert host.dtype == np.uint8 and host.flags.c_contiguous
        assert host.shape[0] >= self.C - self.T and host.shape[1] == self.R
        self.host = host  # a sliding tail writes rows back into it
        out = np.empty(topk.shape[0], dtype=np.int32)
        counts = np.zeros(3, dtype=np.int32)
        args = (self.C, self.S, self.T, self.R, int(self.len[0]),
                self.tok_slot.ctypes.data, self.slot_tok.ctypes.data,
                self.stamp.ctypes.data, self.buf.ctypes.data, host.ctypes.data,
                topk.ctypes.data, int(topk.shape[0]), int(step),
                out.ctypes.data, counts.ctypes.data)
        if self.policy == POLICY_RANDOM:
            err = self.lib.or_resolve_keyed(*args, self.policy, 1 if self.sliding else 0,
                                            1 if alias else 0, self.req, self.seed)
        elif alias:
            err = self.lib.or_resolve_full(*args, self.policy, 1 if self.sliding else 0, 1)
        elif self.sliding:
            err = self.lib.or_resolve_ex(*args, self.policy, 1)
        elif self.policy == POLICY_LRU:
            err = self.lib.or_resolve(*args)
        else:
            err = self.lib.or_resolve_policy(*args, self.policy)
        return out, (int(counts[0]), int(counts[1]), int(counts[2])), int(err)

    def append(self, row: np.ndarray, host: Optional[np.ndarray] = None) -> int:
        """Write the next token's row into the resident tail; returns error bits.

        With a sliding tail, the token leaving the tail is written back into
        ``host`` (uint8 [C-T][R], the request's host rows)."""
        row = np.ascontiguousarray(row, dtype=np.uint8)
        assert row.shape == (self.R,)
        if self.sliding:
            assert host is not None and host.dtype == np.uint8 and host.flags.c_contiguous
            assert host.shape[0] >= self.C - self.T and host.shape[1] == self.R
            return int(self.lib.or_append_sliding(self.C, self.S, self.T, self.R,
                                                  self.len.ctypes.data, self.buf.ctypes.data,
                                                  host.ctypes.data, row.ctypes.data))
        return int(self.lib.or_append(self.C, self.S, self.T, self.R, self.len.ctypes.data,
                                    self.buf.ctypes.data, row.ctypes.data))


def run_request(C: int, S: int, T: int, R: int, host: np.ndarray, topk_rows: np.ndarray,
                length: Optional[int] = None, append_rows: Optional[np.ndarray] = None,
                tail_init: Optional[Callable[[RequestState], None]] = None,
                step0: int = 0, policy: int = POLICY_LRU, sliding: bool = False,
                req: int = 0, seed: int = 0):
    """Replay ``topk_rows`` [steps][K] for one request from the empty state.

    ``append_rows`` [steps][R], when given, is appended before each step's
    resolve (a growing context with a resident tail).  Returns
    (state, out [steps][K], counts [steps][3], resolve error bits [steps]);
    ``state.append_errs`` holds the OR of the appends' error bits.
    """
    st = RequestState(C, S, T, R, length, policy=policy, sliding=sliding, req=req, seed=seed)
    st.append_errs = 0
    if tail_init is not None:
        tail_init(st)
    steps = topk_rows.shape[0]
    outs = np.empty(topk_rows.shape, dtype=np.int32)
    counts = np.empty((steps, 3), dtype=np.int64)
    errs = np.empty(steps, dtype=np.int32)
    for s in range(steps):
        if append_rows is not None:
            st.append_errs |= st.append(append_rows[s], host)
        o, c, e = st.resolve(host, topk_rows[s], step0 + s + 1)
        outs[s] = o
        counts[s] = c
        errs[s] = e
    return st, outs, counts, errs


def parallel_map(fn, items: Sequence, threads: Optional[int] = None):
    """Run ``fn`` over items in threads; results in item order."""
    n = threads or max(1, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(n) as ex:
        return list(ex.map(fn, items))
