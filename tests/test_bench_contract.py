"""bench.py's output contract, on the CPU: the reference arm (the oracle timed
on the host cores) prints one JSON line with the keys the driver reads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_b1_c8k", "--steps", "4", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "impl", "cpu_baseline", "e2e", "config"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 4 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    # the config keys are the ones the GPU arm prints, word for word
    sys.path.insert(0, ROOT)
    import bench
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    assert line["config"] == bench._config(tg.WORKLOADS["tiny_b1_c8k"])


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       timeout=120, cwd=ROOT)
    assert r.returncode != 0


def test_oracle_legs_replay_every_layer_with_appends():
    """The CPU legs run every layer of the sample with a growing context's
    appends, say so in the line, and bound the sample by host memory."""
    import types
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from hierarchical_kv_cache_hs_gb300 import tracegen as tg
    wl = tg.Workload("legs", 77, B=3, C=600, K=40, S=80, T=16, host_ratio=8, layers=2, steps=30,
                     len0=584, grow=1, carry_pct=60, zipf_pct=30, third=tg.THIRD_RECENT, recent=64)
    assert bench._oracle_sample(wl) == [0, 1, 2]
    line = bench.cpu_baseline(wl, types.SimpleNamespace(warmup=3, steps=8), bench.PRIME_STEPS + 11)
    assert line["value"] > 0 and "2 layers" in line["sample"] and "appended" in line["sample"]
    # the big 4-layer workload is sampled to fit the host-memory bound
    big = tg.WORKLOADS["b64_c128k_l4_tail4096"]
    n = len(bench._oracle_sample(big))
    assert 1 <= n < big.B
    assert n * big.layers * big.cold * big.row_bytes <= bench.ORACLE_HOST_BYTES


def test_traffic_figure_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    """roofline.traffic comes from the capture file only while the kernel's
    code still has the fingerprint recorded with the capture."""
    sys.path.insert(0, ROOT)
    import bench
    code = bench._code_fingerprint(bench.KERNEL_SOURCES["hs_resolve_kernel_fused"])
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\nhs_resolve_kernel_fused wl_a 100 20 3000 %s abc1234\n"
                 "hs_resolve_kernel_fused wl_b 100 20 3000 0123456789abcdef abc1234\n" % code)
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    dram, link, note = bench.dram_traffic("hs_resolve_kernel_fused", "wl_a")
    assert (dram, link) == (120, 3000) and "abc1234" in note
    dram, link, note = bench.dram_traffic("hs_resolve_kernel_fused", "wl_b")
    assert dram is None and link is None and note.startswith("stale")
    assert bench.dram_traffic("hs_copy_kernel", "wl_a")[0] is None
    # a comment edit keeps the fingerprint; a code edit changes it
    src = tmp_path / "csrc"
    src.mkdir()
    (src / "k.cu").write_text("int f() { return 1; }  // one\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "hierarchical_kv_cache_hs_gb300", exist_ok=True)
    os.replace(src, tmp_path / "hierarchical_kv_cache_hs_gb300" / "csrc")
    p = tmp_path / "hierarchical_kv_cache_hs_gb300" / "csrc" / "k.cu"
    a = bench._code_fingerprint(["k.cu"])
    p.write_text("/* two */ int f() {\n  return 1;\n}\n")
    assert bench._code_fingerprint(["k.cu"]) == a
    p.write_text("int f() { return 2; }\n")
    assert bench._code_fingerprint(["k.cu"]) != a


def test_traffic_file_matches_the_current_kernels():
    """Every capture on file is either current or reported as stale: the file
    parses, and each row names a known kernel."""
    sys.path.insert(0, ROOT)
    import bench
    rows = [l.split() for l in open(bench.TRAFFIC_FILE) if l.strip() and not l.startswith("#")]
    assert rows
    for r in rows:
        assert len(r) == 7 and r[0] in bench.KERNEL_SOURCES
        assert all(x.isdigit() for x in r[2:5])
