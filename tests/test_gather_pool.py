"""The copy-engine variant's host thread pool, on the CPU.

Thousands of back-to-back batches of varying size: every task of every batch
must run exactly once, and a thread still leaving one batch must not take
part in the next (hs_gather_pool.h claims tasks through a word that carries
the batch number)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "hierarchical_kv_cache_hs_gb300", "csrc")

MAIN = r"""
#include <cstdio>
#include "hs_gather_pool.h"
int main() {
    GatherPool pool(8);
    for (int it = 0; it < 20000; ++it) {
        std::vector<int> hits(1 + it % 37, 0);
        std::function<void(int)> fn = [&](int t) { hits[t] += 1; };
        pool.run((int)hits.size(), fn);
        for (int h : hits)
            if (h != 1) { std::printf("batch %d: a task ran %d times\n", it, h); return 1; }
    }
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_every_task_runs_once_per_batch(tmp_path):
    src = tmp_path / "pool_main.cpp"
    src.write_text(MAIN)
    exe = tmp_path / "pool_main"
    subprocess.run(["g++", "-O2", "-std=c++17", "-pthread", "-I", HDR, str(src), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
