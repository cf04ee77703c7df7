"""The library used from plain C through include/hs.h alone: the example
program compiles and links on any machine, and on a GPU it runs a few
decode steps and checks its own counters and buffer bytes."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "hierarchical_kv_cache_hs_gb300")
SRC = os.path.join(PKG, "examples", "resolve_from_c.c")


def _compile(tmp_path):
    from hierarchical_kv_cache_hs_gb300 import build
    build.build_libhs()
    exe = tmp_path / "resolve_from_c"
    cc = shutil.which("cc") or shutil.which("gcc")
    subprocess.run([cc, "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), SRC, "-L", PKG,
                    "-lhs", "-Wl,-rpath," + PKG, "-o", str(exe)], check=True)
    return exe


@pytest.mark.skipif(shutil.which("cc") is None and shutil.which("gcc") is None, reason="needs a C compiler")
def test_example_compiles_against_the_header(tmp_path):
    assert _compile(tmp_path).exists()


@pytest.mark.gpu
def test_example_runs(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    r = subprocess.run([str(_compile(tmp_path))], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad rows 0" in r.stdout
