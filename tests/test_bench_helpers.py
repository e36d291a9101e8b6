"""Host helpers of bench.py: the device-code hash that keys committed DRAM counters."""
import os
import shutil

import bench


def _copy_tree(tmp_path, kernel):
    rel = bench.KERNEL_SOURCES[kernel]
    dst = tmp_path / rel
    dst.parent.mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, rel), dst)
    (tmp_path / "profiles").mkdir()
    src_prof = os.path.join(bench.ROOT, "profiles", f"{kernel}_training_traffic.txt")
    if os.path.exists(src_prof):
        shutil.copy(src_prof, tmp_path / "profiles")
    return dst


def test_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    kernel = "zl_bwd_main"
    ref = bench.kernel_source_sha256(kernel)
    dst = _copy_tree(tmp_path, kernel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    text = dst.read_text()
    dst.write_text("// a comment line\n" + text.replace("\n#include", "\n/* block\n comment */\n#include", 1))
    assert bench.kernel_source_sha256(kernel) == ref
    dst.write_text(text.replace("namespace zl {", "namespace zl {\nconstexpr int kUnused = 1;", 1))
    assert bench.kernel_source_sha256(kernel) != ref


def test_recorded_traffic_follows_the_device_code(tmp_path, monkeypatch):
    kernel = "zl_bwd_main"
    dst = _copy_tree(tmp_path, kernel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    prof = tmp_path / "profiles" / f"{kernel}_training_traffic.txt"
    prof.write_text(f"dram_bytes_per_launch: 123456\nsource_sha256: {bench.kernel_source_sha256(kernel)}\n")
    assert bench.recorded_traffic(kernel) == 123456.0
    dst.write_text(dst.read_text().replace("namespace zl {", "namespace zl {\nconstexpr int kUnused = 1;", 1))
    assert bench.recorded_traffic(kernel) is None


def test_clock_summary_reads_clock_power_and_reasons():
    lines = ["0, 1942, 2070, 1385.2, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 1900, 2070, 1399.8, 0x4, Not Active, Not Active, Not Active, Active",
             "1, 345, 2070, 60.0, 0x0, Active, Not Active, Not Active, Not Active",  # another GPU
             "garbage"]
    c = bench.summarize_clocks(lines, 0)
    assert c == {"sm_mhz": 1921.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2,
                 "power_w": 1392.5}
    assert bench.summarize_clocks([], 0)["samples"] == 0
