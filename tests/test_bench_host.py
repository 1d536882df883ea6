"""Host-side pieces of bench.py that decide what the JSON line reports: the clock summary, the
peak denominators and the comment-insensitive kernel digest that keeps a DRAM-traffic capture
tied to the code it measured."""
import json
import os

import bench


def test_clock_summary_takes_the_median_and_the_active_reasons():
    lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    c = bench.summarize_clock_lines(lines)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = bench.summarize_clock_lines(["0, 1500, 2070, 1400, 0x8, Active, Not Active, Active, Not Active"])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.summarize_clock_lines([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_peaks_come_from_the_measured_file_or_the_stated_fallback():
    hbm, bf16, src = bench._peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        assert (hbm, bf16, src) == (float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured")
    else:
        assert (hbm, bf16, src) == (6800.0, 1900.0, "fallback")


def test_kernel_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_verify_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    f.write_text("// header\nint a = 1;  // note\n\n/* block\n comment */ int b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_source_digest(["k.cu"])
    f.write_text("// another header\nint a = 1;  // other note\n/* changed */ int b = 2;\n\n\n")
    assert bench.kernel_source_digest(["k.cu"]) == d0
    f.write_text("int a = 1;\nint b = 3;\n")
    assert bench.kernel_source_digest(["k.cu"]) != d0


def test_committed_traffic_capture_names_its_command_and_digest():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for entry in t.values():
        assert entry["command"].startswith("python bench.py")
        assert len(entry["code_sha256"]) == 64
        total = sum(k["dram_read"] + k["dram_write"] for k in entry["kernels"].values())
        assert entry["dram_bytes_per_launch"] == total / entry.get("launches_averaged", 1)


def test_committed_traffic_capture_is_used_only_for_the_code_it_measured():
    """The bench's roofline reports the committed capture while the kernel's code is the code the
    capture measured, and null (stale counters) once it has changed."""
    import json
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    entry = t[bench.HEADLINE_WORKLOAD]
    fresh = entry["code_sha256"] == bench.kernel_source_digest(bench.TC_KERNEL_FILES)
    got = bench._kernel_traffic(bench.TC_KERNEL_FILES, bench.HEADLINE_WORKLOAD)
    assert got == (entry["dram_bytes_per_launch"] if fresh else None)


def test_graph_chunks_cover_exactly_the_requested_steps():
    for n in [1, 2, 3, 5, 20, 63, 64, 65, 100, 127, 128, 129, 2048, 2049]:
        chunks = bench.graph_chunks(n)
        assert sum(g * r for g, r in chunks) == n
        assert all(1 <= g <= bench.GRAPH_MAX and r >= 1 for g, r in chunks)
        assert len(chunks) <= 2
    assert bench.graph_chunks(0) == []
