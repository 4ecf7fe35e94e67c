"""Host-side helpers of bench.py (CPU): the source hash that ties a recorded
DRAM-traffic figure to the code it was measured with, the conversion of an ncu
launch list into that record, and the roofline of the dominant kernel."""

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
        if rec["dram_bytes_per_call"] is not None:  # a whole call was captured
            assert rec["dram_bytes_per_call"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
        for k in rec["per_kernel"].values():  # per-launch records of single kernels
            assert k["launches"] > 0 and k["read_bytes"] >= 0 and k["write_bytes"] >= 0
        got = bench.recorded_traffic(rec["workload"], rec["backward"])
        if rec["kernel_source_hash"] == bench.kernel_source_hash():
            assert got == rec, name
        else:
            assert got is None, name


def _ncu_csv(path, launches):
    """A launch list in the layout of `ncu --csv --metrics ...` (one row per metric)."""
    head = ['"ID"', '"Process ID"', '"Kernel Name"', '"Metric Name"', '"Metric Unit"',
            '"Metric Value"']
    lines = ['==PROF== Connected to process 1', ",".join(head)]
    for i, (name, rd, wr, us) in enumerate(launches):
        for metric, unit, val in (("dram__bytes_read.sum", "Mbyte", rd),
                                  ("dram__bytes_write.sum", "Kbyte", wr),
                                  ("gpu__time_duration.sum", "usecond", us)):
            lines.append(",".join(f'"{x}"' for x in (i, 1, name, metric, unit,
                                                      f"{val:,.2f}")))
    path.write_text("\n".join(lines) + "\n")


def _call(scale):
    return [("void grpo::row_plan_kernel(const unsigned char *, long long, int, int *)",
             0.02, 0.0, 10.0),
            ("void grpo::tc_gemm_kernel<(int)3, (int)2>(CUtensorMap, CUtensorMap, "
             "grpo::TileArgs)", 1000.0 * scale, 800.0, 2000.0),
            ("void at::native::vectorized_elementwise_kernel<4>(int, float)", 5.0, 5.0, 3.0),
            ("void grpo::tc_gemm_kernel<(int)3, (int)2>(CUtensorMap, CUtensorMap, "
             "grpo::TileArgs)", 1000.0 * scale, 800.0, 2000.0),
            ("void grpo::finish_loss_kernel(grpo::FinishArgs)", 0.1, 0.004, 5.0)]


def test_ncu_launch_list_split_into_calls(tmp_path):
    csv = tmp_path / "launches.csv"
    _ncu_csv(csv, _call(1.0) + _call(2.0) + _call(3.0)[:2])  # the last call is cut short
    calls = bench.ncu_calls(str(csv))
    assert len(calls) == 2  # the truncated call is dropped
    for c, scale in zip(calls, (1.0, 2.0)):
        # torch's own kernel is not part of the call; (int) is dropped from names
        assert [d["name"] for d in c] == ["row_plan_kernel", "tc_gemm_kernel<3, 2>",
                                          "tc_gemm_kernel<3, 2>", "finish_loss_kernel"]
        assert c[1]["read"] == 1000.0 * scale * 1e6
        assert c[1]["write"] == 800.0 * 1e3
        assert c[1]["ms"] == 2.0


def test_record_traffic_keeps_the_last_complete_call(tmp_path, monkeypatch):
    csv = tmp_path / "launches.csv"
    _ncu_csv(csv, _call(1.0) + _call(2.0) + _call(3.0)[:2])
    monkeypatch.setattr(bench, "traffic_path",
                        lambda w, b: str(tmp_path / f"traffic_{w}_{b}.json"))
    rec = bench.record_traffic(str(csv), "toy", "stored", "ncu ... python bench.py")
    gemm = rec["per_kernel"]["tc_gemm_kernel<3, 2>"]
    assert gemm["launches"] == 2 and gemm["read_bytes"] == 2 * 2000.0e6
    assert rec["launches_per_call"] == 4
    assert rec["dram_bytes_per_call"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    assert abs(rec["ncu_time_ms_per_call"] - 4.015) < 1e-9
    assert rec["kernel_source_hash"] == bench.kernel_source_hash()
    assert json.loads((tmp_path / "traffic_toy_stored.json").read_text()) == rec


def test_kernel_roofline_takes_the_kernel_with_most_time():
    D, V, valid, calls = 4096, 128256, 16384, 5
    times = [{"name": "row_plan_kernel", "launches": 5, "total_ms": 0.05},
             {"name": "tc_gemm_kernel<3, 2>", "launches": 20, "total_ms": 45.0},
             {"name": "finalize_gform_kernel", "launches": 20, "total_ms": 4.0},
             {"name": "tc_gemm_kernel<2, 2>", "launches": 20, "total_ms": 41.0}]
    peaks = {"hbm_gbs": 7000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1700.0}
    rec = {"per_kernel": {"tc_gemm_kernel<3, 2>": {"launches": 4, "read_bytes": 4.0e9,
                                                   "write_bytes": 2.0e9}}}
    r = bench.kernel_roofline(times, calls, D, V, valid, peaks, rec)
    assert r["kernel"] == "tc_gemm_kernel<3, 2>" and r["bound"] == "tensor"
    assert r["launches_per_call"] == 4 and r["avg_launch_ms"] == 45.0 / 20
    # 2 D V per valid token, over the call's 4 launches of this kernel
    per_launch = 2.0 * D * V * valid / 4
    assert r["algorithmic_flops_per_launch"] == per_launch
    assert abs(r["achieved"] - per_launch / (45.0 / 20 / 1e3) / 1e12) < 1e-9
    # Launches last milliseconds: the burst peak, with the sustained fraction beside it.
    assert r["peak"] == 2000.0 and abs(r["frac"] - r["achieved"] / 2000.0) < 1e-12
    assert abs(r["frac_of_sustained_peak"] - r["achieved"] / 1700.0) < 1e-12
    assert r["traffic"] == 1.5e9
    assert [k["name"] for k in r["per_kernel"]][:2] == ["tc_gemm_kernel<3, 2>",
                                                          "tc_gemm_kernel<2, 2>"]
    assert abs(sum(k["share"] for k in r["per_kernel"]) - 1.0) < 1e-12
    assert all(k["of_call"] is None for k in r["per_kernel"])
    r = bench.kernel_roofline(times, calls, D, V, valid, peaks, rec, call_ms=18.0)
    assert abs(r["per_kernel"][0]["of_call"] - 45.0 / calls / 18.0) < 1e-12
    # A row pass on top is HBM-bound: 4 V bytes per valid token (fp16 logits in,
    # bf16 G out) and 4 bytes per 64-column box (its maximum).
    times[2]["total_ms"] = 99.0
    r = bench.kernel_roofline(times, calls, D, V, valid, peaks, None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 7000.0
    assert r["traffic"] is None
    per_token = 4.0 * V + 4.0 * (-(-V // 64))
    assert abs(r["achieved"] - per_token * valid / 4 / (99.0 / 20 / 1e3) / 1e9) < 1e-9


def test_record_traffic_command_line(tmp_path):
    # The command the profiles give: bench.py --record-traffic <csv> --workload W
    # writes profiles/traffic_W_<backward>.json. Run on a copy of bench.py so the
    # committed profiles stay untouched.
    import shutil
    import subprocess
    import sys

    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, "bench.py"), root / "bench.py")
    shutil.copytree(os.path.join(ROOT, "chunked_log_prob_gb300", "csrc"),
                    root / "chunked_log_prob_gb300" / "csrc")
    csv = tmp_path / "launches.csv"
    _ncu_csv(csv, _call(1.0) + _call(2.0) + _call(3.0)[:2])
    r = subprocess.run([sys.executable, str(root / "bench.py"), "--record-traffic", str(csv),
                        "--workload", "toy", "--backward", "recompute",
                        "--record-command", "ncu ..."],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["workload"] == "toy" and line["launches_per_call"] == 4
    with open(root / "profiles" / "traffic_toy_recompute.json") as f:
        rec = json.load(f)
    assert rec["command"] == "ncu ..." and rec["backward"] == "recompute"
    assert rec["kernel_source_hash"] == bench.kernel_source_hash()
    assert rec["per_kernel"]["tc_gemm_kernel<3, 2>"]["read_bytes"] == 2 * 2000.0e6


def test_record_traffic_of_single_kernel_captures(tmp_path, monkeypatch):
    # A capture of one kernel, a few launches (-k, -c) holds no whole call: the
    # record keeps each kernel's bytes per launch, which is what the roofline reads.
    csv = tmp_path / "one_kernel.csv"
    name = "void grpo::tc_gemm_kernel<(int)3, (int)2>(CUtensorMap, CUtensorMap, grpo::TileArgs)"
    _ncu_csv(csv, [(name, 1000.0, 0.5e6, 2000.0),    # MB read, KB written, us
                   (name, 1200.0, 0.5e6, 2200.0)])
    monkeypatch.setattr(bench, "traffic_path", lambda w, b: str(tmp_path / f"t_{w}_{b}.json"))
    rec = bench.record_traffic(str(csv), "toy", "stored", "ncu -k ...")
    e = rec["per_kernel"]["tc_gemm_kernel<3, 2>"]
    assert e["launches"] == 2 and rec["dram_bytes_per_call"] is None
    assert abs((e["read_bytes"] + e["write_bytes"]) / e["launches"] - 1.6e9) < 1.0
    r = bench.kernel_roofline([{"name": "tc_gemm_kernel<3, 2>", "launches": 4, "total_ms": 8.0}],
                              1, 4096, 128256, 16384, {"hbm_gbs": 7000.0, "bf16_tflops": 2000.0,
                                                       "bf16_tflops_sustained": 1700.0}, rec)
    assert abs(r["traffic"] - 1.6e9) < 1.0
