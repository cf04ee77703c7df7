"""The C-ABI library without a GPU: it loads, exports every entry point that
include/hs.h declares, and its host-side argument checks answer before any
CUDA call (so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hs():
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_libhs()
    from hierarchical_kv_cache_hs_gb300 import hs as mod
    return mod


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(hs_[a-z0-9_]+)\s*\(", text):
            names.append(m.group(1))
    return sorted(set(names))


def test_exports_every_declared_symbol(hs):
    names = _declared_functions()
    assert "hs_create" in names and "hs_resolve" in names and "hs_stats" in names
    lib = ctypes.CDLL(hs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings(hs):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert hs.hs_error_string(code) != "unknown error"
    assert hs.hs_error_string(-99) == "unknown error"


@pytest.mark.parametrize("args,code", [
    ((0, 1024, 1152, 64, 16, 0), -1),        # no requests
    ((4, 0, 1152, 64, 16, 0), -1),           # empty context
    ((4, 1024, 1000, 64, 16, 0), -1),        # row bytes not a multiple of 16
    ((4, 1024, 1152, 0, 16, 0), -1),         # no slots
    ((4, 1024, 1152, 64, 0, 0), -1),         # no host pool
    ((4, 1024, 1152, 64, 16, -1), -1),       # negative tail
    ((4, 1024, 1152, 64, 16, 2048), -1),     # tail longer than the context
    ((4, 1024, 1152, 64, 15, 0), -3),        # 15 * 64 host rows < 1024 cold tokens
    ((5000, 1024, 1152, 64, 16, 0), -6),     # batch beyond the limit
    ((4, 1024, 1152, 20000, 1, 0), -6),      # slots beyond the limit
    ((4, 1024, 1 << 17, 64, 16, 0), -6),     # row beyond the limit
])
def test_create_argument_checks(hs, args, code):
    rc, h = hs.hs_create_rc(*args)
    assert rc == code and not h


def test_null_handle_is_rejected(hs):
    assert hs.hs_resolve_rc(None, 1, 4, 1) == hs.HS_ERR_ARG
    assert hs.lib.hs_stats(None, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_reset(None) == hs.HS_ERR_ARG
    assert hs.hs_host_pool(None) == 0
    assert hs.lib.hs_append(None, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_h2d_read(None, None, 16, 0, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_h2d_read(1, 1, 15, 0, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_reset_requests(None, None, 0, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_resolve_layers_host(None, 1, None, 4, None, None) == hs.HS_ERR_ARG
    assert hs.lib.hs_set_policy(None, hs.HS_POLICY_RANDOM) == hs.HS_ERR_ARG
    assert hs.lib.hs_set_eviction_seed(None, 1) == hs.HS_ERR_ARG
    hs.hs_destroy(None)  # no-op


def test_resolve_layers_host_checks(hs):
    rc = hs.hs_resolve_layers_rc
    assert rc([], [], 4, []) == hs.HS_ERR_ARG
    assert rc([None], [1], 4, [1]) == hs.HS_ERR_ARG
    assert rc([1], [1], 0, [1]) == hs.HS_ERR_ARG
    n = hs.HS_MAX_LAYERS + 1
    assert rc([1] * n, [1] * n, 4, [1] * n) == hs.HS_ERR_LIMIT
    assert hs.lib.hs_resolve_layers(None, 1, None, 4, None, None) == hs.HS_ERR_ARG


PAGES = ("HiSparse blog", "papercache summary", "vLLM Hybrid HiSparse post")


def _declaration_comments():
    """(function name, the last top-level block comment before its declaration)."""
    out = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        blocks = [(m.start(), m.group(0)) for m in re.finditer(r"(?m)^/\*.*?\*/", text, flags=re.S)]
        for m in re.finditer(r"(?m)^(?:const\s+)?[a-z_0-9]+\s*\**\s*(hs_[a-z0-9_]+)\s*\(", text):
            before = [b for start, b in blocks if start < m.start()]
            out.append((m.group(1), before[-1] if before else ""))
    return out


def test_every_declaration_cites_its_passage():
    """Each exported call's comment names the page section that defines the
    operation, or says that no passage does."""
    decls = _declaration_comments()
    assert {"hs_create", "hs_resolve", "hs_stats", "hs_append", "hs_resolve_noalloc"} <= {n for n, _ in decls}
    assert {n for n, _ in decls} == set(_declared_functions())
    for name, comment in decls:
        assert "Source:" in comment, name
        src = comment[comment.index("Source:"):]
        assert "no passage" in src or any(p in src for p in PAGES), name


def test_noalloc_header_states_its_fixed_step():
    """The allocation-free entry point's comment says which step it takes
    (LRU, fixed tail, two launches) and how its set-up and checks behave."""
    comment = dict(_declaration_comments())["hs_resolve_noalloc"]
    flat = " ".join(comment.replace("*", " ").split())
    for phrase in ("LRU eviction", "the fixed resident tail", "two launches", "HS_COPY_SPLIT",
                   "before any stream capture", "tries it again", "16 bytes", "HS_ERR_LIMIT",
                   "race"):
        assert phrase in flat, phrase


def test_noalloc_refuses_misaligned_pointers_without_a_gpu(hs):
    """The alignment checks answer before any CUDA call."""
    args = dict(topk=256, out=512, tok=1024, slot=2048, stamp=4096, lens=8192, pool=16384,
                buf=32768, ctl=65536)

    def call(**over):
        a = dict(args, **over)
        return hs.lib.hs_resolve_noalloc(2, 1024, 64, 128, 1024, 0, a["topk"], 64, a["out"], a["tok"],
                                         a["slot"], a["stamp"], a["lens"], a["pool"], a["buf"],
                                         a["ctl"], None)
    for name, off in (("pool", 8), ("buf", 4), ("ctl", 4), ("topk", 2), ("out", 1), ("tok", 2),
                      ("slot", 2), ("stamp", 2), ("lens", 2)):
        assert call(**{name: args[name] + off}) == hs.HS_ERR_ARG, name


def test_noalloc_binding_checks_torch_arguments(hs):
    """The binding refuses torch tensors of the wrong type, size or layout
    before the call (checked here with CPU tensors; none reaches the library)."""
    torch = pytest.importorskip("torch")
    B, C, S, K, R, H = 2, 1024, 128, 64, 64, 1024
    good = dict(topk_idx=torch.zeros((B, K), dtype=torch.int32),
                out_slot=torch.zeros((B, K), dtype=torch.int32),
                tok_slot=torch.zeros((B, C), dtype=torch.int32),
                slot_tok=torch.zeros((B, S), dtype=torch.int32),
                stamp=torch.zeros((B, S), dtype=torch.int32),
                lengths=torch.zeros(B, dtype=torch.int32),
                host_pool=torch.zeros(B * H * R, dtype=torch.uint8),
                device_buffer=torch.zeros((B, S, R), dtype=torch.uint8),
                control=torch.zeros(8, dtype=torch.int32))
    bad = {"topk_idx": torch.zeros((B, K), dtype=torch.int64),
           "out_slot": torch.zeros((B, K - 1), dtype=torch.int32),
           "tok_slot": torch.zeros((C, B), dtype=torch.int32).t(),
           "stamp": torch.zeros((B, S), dtype=torch.float32),
           "lengths": torch.zeros(B - 1, dtype=torch.int32),
           "device_buffer": torch.zeros((B, S, R - 16), dtype=torch.uint8),
           "control": torch.zeros(7, dtype=torch.int32),
           "host_pool": torch.zeros(B * H * R, dtype=torch.uint8)}  # not pinned
    for name, value in bad.items():
        a = dict(good, **{name: value})
        with pytest.raises(ValueError):
            hs.hs_resolve_noalloc(B, C, R, S, H, 0, a["topk_idx"], K, a["out_slot"], a["tok_slot"],
                                  a["slot_tok"], a["stamp"], a["lengths"], a["host_pool"],
                                  a["device_buffer"], a["control"])


def test_pool_placement_calls_check_their_arguments(hs):
    """The placement switch takes the three modes only; a NULL handle has none."""
    try:
        for mode in (hs.HS_POOL_PAGES_BASE, hs.HS_POOL_PAGES_HUGE, hs.HS_POOL_PAGES_AUTO):
            assert hs.lib.hs_set_host_pool_pages(mode) == 0
        assert hs.lib.hs_set_host_pool_pages(3) == hs.HS_ERR_ARG
        assert hs.lib.hs_set_host_pool_pages(-1) == hs.HS_ERR_ARG
    finally:
        hs.lib.hs_set_host_pool_pages(hs.HS_POOL_PAGES_AUTO)
    assert hs.lib.hs_host_pool_pages(None) == hs.HS_ERR_ARG
    assert hs.hs_huge_page_bytes() >= 0
