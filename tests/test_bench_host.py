"""Host-side helpers of bench.py (CPU): the source hash that ties a recorded
DRAM-traffic figure to the code it was measured with, and the JSON keys the
benchmark line must carry."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_tokens_drop_comments_and_layout_only():
    src = ('int a = 1;  // note\n/* block\n   comment */ const char* s = "// kept";\n'
           "char q = '\"';  float b = a /* inline */ * 2;\n")
    got = bench.code_tokens(src)
    assert got == 'int a = 1; const char* s = "// kept"; char q = \'"\'; float b = a * 2;'
    # Code changes still change the tokens.
    assert bench.code_tokens(src.replace("a = 1", "a = 2")) != got


def test_recorded_traffic_is_used_only_for_its_own_code():
    # A committed record is reported while the code matches its hash, and
    # null otherwise; its byte counts are self-consistent.
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        if not (name.startswith("traffic_") and name.endswith(".json")):
            continue
        with open(os.path.join(ROOT, "profiles", name)) as f:
            rec = json.load(f)
        assert rec["dram_bytes_per_call"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
        got = bench.recorded_traffic(rec["workload"], rec["backward"])
        if rec["kernel_source_hash"] == bench.kernel_source_hash():
            assert got == rec["dram_bytes_per_call"], name
        else:
            assert got is None, name
