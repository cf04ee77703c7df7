"""The resolve kernel's shared-memory layout, checked on the host for every
top-k size: the header's size functions compiled by the host compiler (no
GPU), so a layout that would misalign the kernel's 16-byte copies or exceed
the per-block shared memory is caught before any launch."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hierarchical_kv_cache_hs_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r"""
#include <cstdio>
#include "hs_internal.h"

// Largest shared memory one block may use on sm_103a (opt-in), less the
// kernel's static arrays (a few hundred bytes; 1 KB kept free).
static const size_t kLimit = 227u * 1024u - 1024u;

int main()
{
    for (int K = 1; K <= HS_MAX_TOPK; ++K) {
        const int bits = hs_hash_bits(K);
        const int A = hs_resolve_region_a_ints(bits, K);
        if ((1 << bits) < 2 * K) { printf("K=%d: hash more than half full\n", K); return 1; }
        if (A % 4 != 0) { printf("K=%d: region A of %d ints misaligns the stamp row\n", K, A); return 1; }
        if (A < (2 << bits)) { printf("K=%d: region A smaller than the hash\n", K); return 1; }
        const int E = (K + HS_RESOLVE_THREADS - 1) / HS_RESOLVE_THREADS;
        if (2 * A < 2 * (HS_AGE_SUBHIST * HS_AGE_BINS + E * HS_RESOLVE_THREADS) + K) {
            printf("K=%d: region A smaller than histograms + out values + copy list\n", K);
            return 1;
        }
        const int Ss[] = {K, K + 1, K + 2, K + 3, HS_MAX_SLOTS};
        for (int S : Ss) {
            if (S > HS_MAX_SLOTS) continue;
            const size_t bytes = hs_resolve_base_bytes(K, S, bits);
            if (bytes > kLimit) { printf("K=%d S=%d: %zu bytes\n", K, S, bytes); return 1; }
        }
    }
    printf("ok\n");
    return 0;
}
"""


def test_resolve_shared_memory_layout(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "layout.cpp"
    exe = tmp_path / "layout"
    src.write_text(PROGRAM)
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", INCLUDE, "-I", CUDA_INC,
                        str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
