"""Python binding of ``libhs.so`` (the C ABI in ``include/hs.h``).

Argument marshalling only: every step of the swap-in path runs in the CUDA
library.  Pointers may be given as integers, torch tensors (``data_ptr()``) or
numpy arrays; streams as ``None`` (legacy default stream), an integer handle
or a ``torch.cuda.Stream``.  Errors returned by the library raise ``HsError``.

Importing this module loads the library and raises ``ImportError`` when it has
not been built -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhs.so")

HS_OK = 0
HS_ERR_ARG = -1
HS_ERR_TOPK_GT_SLOTS = -2
HS_ERR_CAPACITY = -3
HS_ERR_ALLOC = -4
HS_ERR_CUDA = -5
HS_ERR_LIMIT = -6

HS_E_RANGE = 1
HS_E_DUP = 2
HS_E_APPEND = 4
HS_E_STATE = 8

HS_TAIL_FIXED = 0
HS_TAIL_SLIDING = 1

HS_POLICY_LRU = 0
HS_POLICY_FIFO = 1
HS_POLICY_RANDOM = 2

HS_COPY_AUTO = 0
HS_COPY_FUSED = 1
HS_COPY_SPLIT = 2
HS_COPY_CLUSTER = 3
HS_MAX_CLUSTER = 16
HS_CLUSTER_WIDE_BATCH = 4
HS_CLUSTER_MAX_BATCH = 128
HS_MAX_COPY_CTAS = 65535
HS_POOL_PAGES_AUTO = 0
HS_POOL_PAGES_BASE = 1
HS_POOL_PAGES_HUGE = 2
HS_POOL_HUGE_MIN_BYTES = 1 << 34
HS_FUSED_MIN_BATCH = 16
HS_FUSED_MAX_REQUEST_BYTES = 1 << 20

HS_MAX_TOPK = 4096
HS_MAX_SLOTS = 16384
HS_MAX_BATCH = 4096
HS_MAX_ROW_BYTES = 65536
HS_MAX_LAYERS = 16


class HsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%d)" % (where, hs_error_string(code), code))


class hs_stats_t(ctypes.Structure):
    _fields_ = [
        ("steps", ctypes.c_int64),
        ("hits", ctypes.c_int64),
        ("misses", ctypes.c_int64),
        ("inplace", ctypes.c_int64),
        ("bytes_copied", ctypes.c_int64),
        ("err_bits", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libhs.so is not built (run __graft_entry__.build() or "
                          "python -m hierarchical_kv_cache_hs_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "hs_create": ([I, I, I, I, I, I, ctypes.POINTER(P)], I),
        "hs_destroy": ([P], None),
        "hs_resolve": ([P, P, I, P, P], I),
        "hs_resolve_host": ([P, P, I, P, P], I),
        "hs_resolve_multi": ([P, P, I, I, P, P], I),
        "hs_resolve_layers": ([P, I, P, I, P, P], I),
        "hs_resolve_layers_host": ([P, I, P, I, P, P], I),
        "hs_resolve_ce": ([P, P, I, P, P], I),
        "hs_stats": ([P, ctypes.POINTER(hs_stats_t), P], I),
        "hs_host_pool": ([P], P),
        "hs_host_pool_bytes": ([P], Z),
        "hs_set_host_pool_pages": ([I], I),
        "hs_host_pool_pages": ([P], I),
        "hs_huge_page_bytes": ([], Z),
        "hs_device_buffer": ([P], P),
        "hs_device_buffer_bytes": ([P], Z),
        "hs_set_lengths": ([P, P], I),
        "hs_append": ([P, P, P], I),
        "hs_set_tail_rows": ([P, I, I, I, P], I),
        "hs_export_state": ([P, P, P, P, P], I),
        "hs_export_buffer": ([P, I, P], I),
        "hs_import_state": ([P, P, P, P, I], I),
        "hs_reset": ([P], I),
        "hs_reset_requests": ([P, P, I, P, P], I),
        "hs_h2d_read": ([P, P, Z, I, P], I),
        "hs_profile_events": ([P, P, P], I),
        "hs_set_copy_mode": ([P, I], I),
        "hs_set_cluster_size": ([P, I], I),
        "hs_set_copy_ctas": ([P, I], I),
        "hs_cluster_size": ([P], I),
        "hs_launch_mode": ([P], I),
        "hs_resolve_launches": ([P], I),
        "hs_set_policy": ([P, I], I),
        "hs_set_eviction_seed": ([P, ctypes.c_uint64], I),
        "hs_set_tail_mode": ([P, I], I),
        "hs_resolve_noalloc": ([I, I, I, I, I, I, P, I, P, P, P, P, P, P, P, P, P], I),
        "hs_error_string": ([I], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError("cannot take a pointer of %r" % type(x))


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError("cannot take a stream handle of %r" % type(s))


def _check(rc: int, where: str) -> None:
    if rc != HS_OK:
        raise HsError(rc, where)


def hs_error_string(code: int) -> str:
    return lib.hs_error_string(int(code)).decode()


def hs_create(batch: int, ctx_len: int, row_bytes: int, buffer_slots: int, host_ratio: int,
              resident_tail: int = 0) -> int:
    """Create a handle; returns its address.  Raises HsError on a library error."""
    out = ctypes.c_void_p()
    _check(lib.hs_create(batch, ctx_len, row_bytes, buffer_slots, host_ratio, resident_tail,
                         ctypes.byref(out)), "hs_create")
    return out.value


def hs_create_rc(batch, ctx_len, row_bytes, buffer_slots, host_ratio, resident_tail=0):
    """hs_create returning (code, handle) instead of raising."""
    out = ctypes.c_void_p()
    rc = lib.hs_create(batch, ctx_len, row_bytes, buffer_slots, host_ratio, resident_tail,
                       ctypes.byref(out))
    return rc, out.value


def hs_destroy(h: int) -> None:
    lib.hs_destroy(h)


def hs_resolve(h: int, topk_idx, K: int, out_slot, stream=None) -> None:
    _check(lib.hs_resolve(h, _ptr(topk_idx), int(K), _ptr(out_slot), _stream(stream)),
           "hs_resolve")


def _ptr_array(xs):
    arr = (ctypes.c_void_p * max(len(xs), 1))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def hs_resolve_layers_rc(handles, topk_idx, K: int, out_slot, stream=None) -> int:
    """handles, topk_idx and out_slot: sequences of L entries (one per layer)."""
    L = len(handles)
    if len(topk_idx) != L or len(out_slot) != L:
        return HS_ERR_ARG
    return lib.hs_resolve_layers(_ptr_array(handles), L, _ptr_array(topk_idx), int(K),
                                 _ptr_array(out_slot), _stream(stream))


def hs_resolve_layers(handles, topk_idx, K: int, out_slot, stream=None) -> None:
    """L independent layers' step in one launch; same results as hs_resolve per layer."""
    _check(hs_resolve_layers_rc(handles, topk_idx, K, out_slot, stream), "hs_resolve_layers")


def hs_resolve_layers_host(handles, topk_idx, K: int, out_slot, stream=None) -> None:
    """hs_resolve_layers from host buffers (sequences of L addresses or arrays); synchronous."""
    L = len(handles)
    if len(topk_idx) != L or len(out_slot) != L:
        raise HsError(HS_ERR_ARG, "hs_resolve_layers_host")
    _check(lib.hs_resolve_layers_host(_ptr_array(handles), L, _ptr_array(topk_idx), int(K),
                                      _ptr_array(out_slot), _stream(stream)),
           "hs_resolve_layers_host")


def hs_resolve_rc(h: int, topk_idx, K: int, out_slot, stream=None) -> int:
    return lib.hs_resolve(h, _ptr(topk_idx), int(K), _ptr(out_slot), _stream(stream))


def hs_resolve_multi(h: int, topk_idx, P: int, K: int, out_slot, stream=None) -> None:
    """P draft positions' top-k rows ([B][P][K]) resolved together."""
    _check(lib.hs_resolve_multi(h, _ptr(topk_idx), int(P), int(K), _ptr(out_slot),
                                _stream(stream)), "hs_resolve_multi")


def hs_resolve_host(h: int, topk_idx, K: int, out_slot, stream=None) -> None:
    _check(lib.hs_resolve_host(h, _ptr(topk_idx), int(K), _ptr(out_slot), _stream(stream)),
           "hs_resolve_host")


def hs_resolve_ce(h: int, topk_idx, K: int, out_slot, stream=None) -> None:
    """The copy-engine comparison variant (synchronises once per call)."""
    _check(lib.hs_resolve_ce(h, _ptr(topk_idx), int(K), _ptr(out_slot), _stream(stream)),
           "hs_resolve_ce")


def hs_stats(h: int, last_miss=None) -> dict:
    st = hs_stats_t()
    _check(lib.hs_stats(h, ctypes.byref(st), _ptr(last_miss)), "hs_stats")
    return {f: getattr(st, f) for f, _ in hs_stats_t._fields_ if f != "reserved"}


def hs_host_pool(h: int) -> int:
    return lib.hs_host_pool(h) or 0


def hs_host_pool_bytes(h: int) -> int:
    return int(lib.hs_host_pool_bytes(h))


def hs_set_host_pool_pages(mode: int) -> None:
    """Placement of the host pools of handles created from now on (HS_POOL_PAGES_*)."""
    _check(lib.hs_set_host_pool_pages(int(mode)), "hs_set_host_pool_pages")


def hs_host_pool_pages(h: int) -> int:
    r = lib.hs_host_pool_pages(h)
    if r < 0:
        raise HsError(r, "hs_host_pool_pages")
    return int(r)


def hs_huge_page_bytes() -> int:
    return int(lib.hs_huge_page_bytes())


def hs_device_buffer(h: int) -> int:
    return lib.hs_device_buffer(h) or 0


def hs_device_buffer_bytes(h: int) -> int:
    return int(lib.hs_device_buffer_bytes(h))


def hs_set_lengths(h: int, lengths) -> None:
    arr = np.ascontiguousarray(lengths, dtype=np.int32)
    _check(lib.hs_set_lengths(h, arr.ctypes.data), "hs_set_lengths")


def hs_append(h: int, rows_dev, stream=None) -> None:
    _check(lib.hs_append(h, _ptr(rows_dev), _stream(stream)), "hs_append")


def hs_set_tail_rows(h: int, b: int, first_token: int, rows_host: np.ndarray) -> None:
    arr = np.ascontiguousarray(rows_host, dtype=np.uint8)
    _check(lib.hs_set_tail_rows(h, int(b), int(first_token), int(arr.shape[0]), arr.ctypes.data),
           "hs_set_tail_rows")


def hs_export_state(h: int, tok_slot=None, slot_tok=None, stamp=None) -> int:
    """Copy the tables into the given host arrays; returns the step counter."""
    step = np.zeros(1, dtype=np.int32)
    _check(lib.hs_export_state(h, _ptr(tok_slot), _ptr(slot_tok), _ptr(stamp), step.ctypes.data),
           "hs_export_state")
    return int(step[0])


def hs_import_state(h: int, tok_slot, slot_tok, stamp, step: int) -> None:
    """Load a saved state (host arrays as hs_export_state writes them)."""
    a = np.ascontiguousarray(tok_slot, dtype=np.int32)
    b = np.ascontiguousarray(slot_tok, dtype=np.int32)
    c = np.ascontiguousarray(stamp, dtype=np.int32)
    _check(lib.hs_import_state(h, a.ctypes.data, b.ctypes.data, c.ctypes.data, int(step)),
           "hs_import_state")


def hs_import_state_rc(h: int, tok_slot, slot_tok, stamp, step: int) -> int:
    a = np.ascontiguousarray(tok_slot, dtype=np.int32)
    b = np.ascontiguousarray(slot_tok, dtype=np.int32)
    c = np.ascontiguousarray(stamp, dtype=np.int32)
    return lib.hs_import_state(h, a.ctypes.data, b.ctypes.data, c.ctypes.data, int(step))


def hs_export_buffer(h: int, b: int, dst_host) -> None:
    _check(lib.hs_export_buffer(h, int(b), _ptr(dst_host)), "hs_export_buffer")


def hs_reset(h: int) -> None:
    _check(lib.hs_reset(h), "hs_reset")


def hs_reset_requests(h: int, req_ids, n: int, lengths=None, stream=None) -> None:
    """Empty the state of the n requests listed in req_ids (device int32 [n]),
    with new lengths (device int32 [n]) or C; asynchronous on `stream`."""
    _check(lib.hs_reset_requests(h, _ptr(req_ids), int(n), _ptr(lengths), _stream(stream)),
           "hs_reset_requests")


def hs_h2d_read(src_host, dst_dev, nbytes: int, blocks: int = 0, stream=None) -> None:
    _check(lib.hs_h2d_read(_ptr(src_host), _ptr(dst_dev), int(nbytes), int(blocks),
                           _stream(stream)), "hs_h2d_read")


HS_NOALLOC_MAX_ENTRIES = 524288


def _check_buffer(x, name, dtype, numel, device=None, pinned=False):
    """Shape, type and placement of one torch tensor argument of
    hs_resolve_noalloc (the library cannot see the sizes of caller buffers).
    Raw addresses are passed through: their sizes are the caller's to keep."""
    if x is None:
        raise ValueError("%s is required" % name)
    if not hasattr(x, "data_ptr") or not hasattr(x, "is_contiguous"):
        return
    if x.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, x.dtype))
    if not x.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if x.numel() < numel:
        raise ValueError("%s holds %d elements, needs %d" % (name, x.numel(), numel))
    if device is not None and x.device != device:
        raise ValueError("%s must be on %s, is on %s" % (name, device, x.device))
    if pinned and not (x.device.type == "cpu" and x.is_pinned()):
        raise ValueError("%s must be pinned host memory" % name)


def hs_resolve_noalloc(batch, ctx_len, row_bytes, buffer_slots, host_rows, resident_tail,
                       topk_idx, K, out_slot, tok_slot, slot_tok, stamp, lengths, host_pool,
                       device_buffer, control, stream=None) -> None:
    """The swap-in step on caller-owned state; the library allocates nothing.

    For callers that cannot let a library allocate device memory (an engine
    that reserved HBM for its own pool, a loop where an allocation would stall
    the device).  ``control`` is a zeroed 32-byte device block (hs_control_t).
    Torch tensors are checked here (dtype, contiguity, size, device, pinned
    pool) and a mismatch raises ValueError before the call.
    """
    import torch
    B, C, R, S, T, K = (int(batch), int(ctx_len), int(row_bytes), int(buffer_slots),
                        int(resident_tail), int(K))
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else None
    i32, u8 = torch.int32, torch.uint8
    _check_buffer(topk_idx, "topk_idx", i32, B * K, dev)
    _check_buffer(out_slot, "out_slot", i32, B * K, dev)
    _check_buffer(tok_slot, "tok_slot", i32, B * C, dev)
    _check_buffer(slot_tok, "slot_tok", i32, B * S, dev)
    _check_buffer(stamp, "stamp", i32, B * S, dev)
    _check_buffer(lengths, "lengths", i32, B, dev)
    _check_buffer(device_buffer, "device_buffer", u8, B * (S + T) * R, dev)
    if hasattr(control, "element_size"):
        _check_buffer(control, "control", control.dtype, -(-32 // control.element_size()), dev)
    _check_buffer(host_pool, "host_pool", u8, B * int(host_rows) * R, pinned=True)
    _check(lib.hs_resolve_noalloc(B, C, R, S, int(host_rows), T, _ptr(topk_idx), K,
                                  _ptr(out_slot), _ptr(tok_slot), _ptr(slot_tok), _ptr(stamp),
                                  _ptr(lengths), _ptr(host_pool), _ptr(device_buffer),
                                  _ptr(control), _stream(stream)), "hs_resolve_noalloc")


def hs_set_copy_mode(h: int, mode: int) -> None:
    _check(lib.hs_set_copy_mode(h, int(mode)), "hs_set_copy_mode")


def hs_set_copy_ctas(h: int, n: int) -> None:
    """CTAs of the split mode's copy kernel (0 = the default grid)."""
    _check(lib.hs_set_copy_ctas(h, int(n)), "hs_set_copy_ctas")


def hs_set_cluster_size(h: int, n: int) -> None:
    """CTAs per request in cluster mode (0 = the handle's default)."""
    _check(lib.hs_set_cluster_size(h, int(n)), "hs_set_cluster_size")


def hs_cluster_size(h: int) -> int:
    n = lib.hs_cluster_size(h)
    if n < 0:
        raise HsError(n, "hs_cluster_size")
    return n


def hs_launch_mode(h: int) -> int:
    """HS_COPY_FUSED, HS_COPY_SPLIT or HS_COPY_CLUSTER: what the next hs_resolve launches."""
    n = lib.hs_launch_mode(h)
    if n < 0:
        raise HsError(n, "hs_launch_mode")
    return n


def hs_set_tail_mode(h: int, mode: int) -> None:
    _check(lib.hs_set_tail_mode(h, int(mode)), "hs_set_tail_mode")


def hs_set_policy(h: int, policy: int) -> None:
    _check(lib.hs_set_policy(h, int(policy)), "hs_set_policy")


def hs_set_eviction_seed(h: int, seed: int) -> None:
    """Seed of HS_POLICY_RANDOM's keys (64 bits)."""
    _check(lib.hs_set_eviction_seed(h, int(seed) & ((1 << 64) - 1)), "hs_set_eviction_seed")


def hs_resolve_launches(h: int) -> int:
    n = lib.hs_resolve_launches(h)
    if n < 0:
        raise HsError(n, "hs_resolve_launches")
    return n


def hs_profile_events(h: int, before_copy=None, after_copy=None) -> None:
    """Record two CUDA events (torch.cuda.Event or raw handles) around the copy kernel."""
    def ev(e):
        if e is None:
            return None
        return e.cuda_event if hasattr(e, "cuda_event") else int(e)
    _check(lib.hs_profile_events(h, ev(before_copy), ev(after_copy)), "hs_profile_events")


class Handle:
    """Owning wrapper: one swap-in state (one layer, B requests)."""

    def __init__(self, batch, ctx_len, row_bytes, buffer_slots, host_ratio, resident_tail=0):
        self.B, self.C, self.R, self.S = batch, ctx_len, row_bytes, buffer_slots
        self.T, self.host_ratio = resident_tail, host_ratio
        self.H = host_ratio * buffer_slots
        self.h = hs_create(batch, ctx_len, row_bytes, buffer_slots, host_ratio, resident_tail)

    def close(self):
        if getattr(self, "h", None):
            hs_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def host_pool(self) -> np.ndarray:
        """The pinned host pool as a numpy view [B][H][R] (uint8)."""
        n = hs_host_pool_bytes(self.h)
        buf = (ctypes.c_uint8 * n).from_address(hs_host_pool(self.h))
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.B, self.H, self.R)

    def resolve(self, topk_idx, K, out_slot, stream=None):
        hs_resolve(self.h, topk_idx, K, out_slot, stream)

    def stats(self, last_miss=None):
        return hs_stats(self.h, last_miss)

    def export_state(self):
        tok = np.empty((self.B, self.C), dtype=np.int32)
        st = np.empty((self.B, self.S), dtype=np.int32)
        stamp = np.empty((self.B, self.S), dtype=np.int32)
        step = hs_export_state(self.h, tok, st, stamp)
        return tok, st, stamp, step

    def export_buffer(self, b: int) -> np.ndarray:
        out = np.empty((self.S + self.T, self.R), dtype=np.uint8)
        hs_export_buffer(self.h, b, out)
        return out
