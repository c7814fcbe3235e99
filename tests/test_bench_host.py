"""Host logic of bench.py that needs no GPU: the code hash that ties a committed ncu traffic
capture to the kernel sources it measured, and the shape of that capture's record."""
import json
import os
import shutil

import bench


def test_code_tokens_drops_comments_and_layout():
    src = "int a = 1;   // note\n/* block\n comment */ float b =\n\t2.0f; // end"
    assert bench.code_tokens(src) == "int a = 1; float b = 2.0f;"


def test_code_tokens_keeps_literals():
    src = 'asm("mov.u32 %0, 1; // not a comment /* nor this */" : "=r"(x)); char q = \'"\'; char e = \'\\\'\';'
    out = bench.code_tokens(src)
    assert '"mov.u32 %0, 1; // not a comment /* nor this */"' in out
    assert "'\"'" in out and "'\\''" in out


def _copy_sources(tmp_path):
    dst = tmp_path / "comm_overlapped_gemm_gb300" / "csrc"
    dst.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "comm_overlapped_gemm_gb300", "csrc")
    for name in bench.FUSED_KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    return dst


def test_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_source_hash()
    f = dst / "tdx_kernel.cuh"
    text = f.read_text()
    f.write_text(text + "\n// a comment added at the end\n/* and a block */\n")
    assert bench.kernel_source_hash() == base
    f.write_text(text + "\nstatic constexpr int kUnused = 1;\n")
    assert bench.kernel_source_hash() != base


def test_traffic_record_is_consistent():
    path = os.path.join(bench.ROOT, "profiles", "tdx_fused_rs_w8_traffic.json")
    with open(path) as fh:
        d = json.load(fh)
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_written"]
    assert d["algorithmic_bytes_per_launch"] > 0
    assert "--clock-control none" in d["command"]
    assert len(d["kernel_source_sha256"]) == 64


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the CPU oracle on a bounded sample of the same workload and
    prints one JSON line with the main arm's metric, unit and direction, a `cpu_baseline` that
    describes the run and a zero-copy `e2e`."""
    import subprocess
    import sys
    res = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         cwd=bench.ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_peak_follows_the_length_of_the_timed_region():
    pk = {"bf16_tflops": 1915.0, "bf16_tflops_sustained": 1713.0}
    v, src = bench.bf16_peak(pk, "measured", 0.05)
    assert v == 1915.0 and "burst" in src
    v, src = bench.bf16_peak(pk, "measured", 4.0)
    assert v == 1713.0 and "sustained" in src
    v, _ = bench.bf16_peak({"bf16_tflops": 1900.0}, "fallback", 4.0)
    assert v == 1900.0


def test_clock_samples_stay_out_of_the_repository(monkeypatch, tmp_path):
    monkeypatch.setenv("TDX_CLOCKS_DIR", str(tmp_path))
    c = bench.ClockSampler(0)
    assert c.path.startswith(str(tmp_path))
    monkeypatch.delenv("TDX_CLOCKS_DIR")
    assert not bench.ClockSampler(0).path.startswith(bench.ROOT)
