"""Host-side pieces of bench.py that decide what its JSON line reports (no GPU)."""
from pathlib import Path

import bench

CSRC = Path(bench.__file__).resolve().parent / "paged_kv_cache_11_gb300" / "csrc"


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // trailing\n\n/* block\n comment */int b;\n  // whole line\nint c;  \n"
    assert bench._code_only(src) == "int a;\nint b;\nint c;"


def test_comment_edits_keep_the_code_hash_and_code_edits_change_it():
    text = (CSRC / "decode.cu").read_text()
    base = bench._code_only(text)
    assert bench._code_only(text.replace("// Grid:", "// The grid:", 1)) == base
    assert bench._code_only(text + "\n/* a note */\n") == base
    assert bench._code_only(text.replace("const int tid = threadIdx.x", "const int tid = (int)threadIdx.x", 1)) != base


def test_traffic_figure_is_reported_only_for_the_code_it_was_taken_on():
    """A traffic entry is used when its key is the current decode code's hash,
    and ignored (the bench line reports null) otherwise."""
    lines = [l.split() for l in bench.TRAFFIC_FILE.read_text().splitlines() if l and not l.startswith("#")]
    assert lines and all(len(l) == 3 for l in lines)
    assert bench.decode_source_hash(grouped=True) != bench.decode_source_hash()
    for workload, key, value in lines:
        h = bench.decode_source_hash(grouped=workload.endswith("_grouped"))
        got = bench.traffic_per_launch(workload)
        assert (got is not None) == (key == h), (workload, key, h)
        if got is not None:
            assert got == float(value)
    assert bench.traffic_per_launch("no_such_workload") is None


def test_percentiles_and_clock_summary():
    p = bench.percentiles([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0, 9.0, 10.0, 11.0])
    assert p["median_ms"] == 6.0 and p["n"] == 11 and p["p10_ms"] == 2.0 and p["p90_ms"] == 10.0
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbage"]
    c = bench.ClockSampler.summarise(rows)
    assert c == {"sm_mhz": 2025.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}
    assert bench.ClockSampler.summarise(["garbage"]) is None


def test_default_run_measures_the_long_context_layer_and_the_8b_layer():
    a = bench.parse_args([])
    assert a.workload == "llama70b_long" and a.extra is None
