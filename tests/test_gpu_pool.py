"""The host pool's placement on the host, read back from the kernel's view of
this process: a huge-page pool is one mapping advised for huge pages, left out
of forked children, and (where the device names a host NUMA node) preferring
that node; a cudaHostAlloc pool is none of those."""
import os
import re

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_all()


def _vma(addr, path="/proc/self/smaps"):
    """The lines of the mapping that holds addr, from smaps or numa_maps."""
    lines = open(path).read().splitlines()
    for i, line in enumerate(lines):
        head = line.split()[0]
        if path.endswith("numa_maps"):
            if int(head, 16) == addr:
                return [line]
            continue
        if "-" in head and not line.startswith(" "):
            lo, hi = (int(x, 16) for x in head.split("-"))
            if lo <= addr < hi:
                out = [line]
                for nxt in lines[i + 1:]:
                    if "-" in nxt.split()[0] and ":" not in nxt.split()[0]:
                        break
                    out.append(nxt)
                return out
    return None


def _flags(vma):
    for line in vma:
        if line.startswith("VmFlags:"):
            return line.split()[1:]
    return []


@pytest.mark.parametrize("placement", ["base", "huge"])
def test_pool_mapping(placement):
    from hierarchical_kv_cache_hs_gb300 import hs
    want = hs.HS_POOL_PAGES_BASE if placement == "base" else hs.HS_POOL_PAGES_HUGE
    hp = hs.hs_huge_page_bytes()
    if want == hs.HS_POOL_PAGES_HUGE and hp == 0:
        pytest.skip("the host offers no transparent huge pages")
    hs.hs_set_host_pool_pages(want)
    try:
        h = hs.Handle(2, 4096, 1152, 256, 16, 0)
    finally:
        hs.hs_set_host_pool_pages(hs.HS_POOL_PAGES_AUTO)
    try:
        assert hs.hs_host_pool_pages(h.h) == want
        pool, n = hs.hs_host_pool(h.h), hs.hs_host_pool_bytes(h.h)
        vma = _vma(pool)
        assert vma is not None
        flags = _flags(vma)
        if want == hs.HS_POOL_PAGES_HUGE:
            assert pool % hp == 0  # aligned to the huge-page size
            assert "hg" in flags and "dc" in flags, flags
            lo, hi = (int(x, 16) for x in vma[0].split()[0].split("-"))
            assert hi - lo >= n
            # the policy is the default (the device names no host node) or a
            # preference for one online node
            if os.path.exists("/proc/self/numa_maps"):
                nm = _vma(lo, "/proc/self/numa_maps")
                assert nm is not None
                # "prefer:N", or "prefer (many):N" on kernels that show a
                # single-node preference that way
                m = re.match(r"[0-9a-f]+ (default|prefer(?: \(many\))?:(\d+))( |$)", nm[0])
                assert m, nm[0]
                if m.group(2) is not None:
                    assert os.path.exists("/sys/devices/system/node/node%s" % m.group(2))
        else:
            assert "hg" not in flags
        # the pool is written and read back through the host pointer either way
        view = h.host_pool()
        view[1, 7, :] = 0xA5
        assert int(view[1, 7, 100]) == 0xA5
    finally:
        h.close()
