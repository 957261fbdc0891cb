"""Host-side logic of bench.py, no GPU: the algorithmic work the roofline divides by, the
traffic record's tie to the kernel sources, and the reference arm's JSON line."""
import json
import os
import shutil
import subprocess
import sys

import bench
from mixture_experts_layer_scores_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = synth.CONFIGS


def test_algorithmic_work_matches_closed_forms():
    # handbook layer: R = N k = 65536 rows of D = 2048, F = 1024, bf16
    a = bench.algorithmic(C["handbook"])
    assert a["gemm_flops"] == 6 * 65536 * 2048 * 1024                    # 824.6 GFLOP
    assert a["combine_bytes"] == 65536 * 2048 * 2 + 8 * 65536 + 2 * 8192 * 2048 * 2  # 336.1 MB
    assert a["permute_bytes"] == 12 * 65536                                # gathering: ids only
    copy = bench.algorithmic(C["handbook"], copy_rows=True)
    assert copy["permute_bytes"] == 8192 * 2048 * 2 + 65536 * 2048 * 2 + 12 * 65536  # 302.8 MB
    assert a["router_flops"] == 2 * 8192 * 2048 * 64
    # DeepSeek-V3 shape: the shared expert's row joins the combine
    d = bench.algorithmic(C["deepseek_v3"])
    assert d["combine_bytes"] == 32768 * 7168 * 2 + 8 * 32768 + 3 * 4096 * 7168 * 2  # 646.2 MB
    assert d["shared_flops"] == 6 * 4096 * 7168 * 2048


SRCS = ["mixture_experts_layer_scores_b300/csrc/grouped_swiglu.cu",
        "mixture_experts_layer_scores_b300/csrc/tc_common.cuh",
        "mixture_experts_layer_scores_b300/csrc/moe_internal.cuh"]


def _tree(tmp, alter=None):
    """A copy of the GEMM sources with traffic records written for them (hash of the copies),
    then optionally one source changed after the records were taken."""
    import hashlib
    for rel in SRCS:
        dst = os.path.join(tmp, rel)
        os.makedirs(os.path.dirname(dst), exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), dst)
    h = hashlib.sha256()
    for rel in SRCS:
        with open(os.path.join(tmp, rel), "rb") as f:
            h.update(f.read())
    os.makedirs(os.path.join(tmp, "profiles"), exist_ok=True)
    for suffix, nbytes in (("", 1500000000), ("_gather", 1400000000)):
        with open(os.path.join(tmp, "profiles", f"grouped_gemm_handbook{suffix}_traffic.txt"), "w") as f:
            f.write(f"# test record\nsources={' '.join(SRCS)}\nsources_sha256={h.hexdigest()}\n"
                    f"dram_bytes_per_call={nbytes}\n")
    if alter:
        with open(os.path.join(tmp, alter), "a") as f:
            f.write("\n// changed\n")


def test_traffic_record_holds_only_for_the_recorded_sources(tmp_path, monkeypatch):
    same, changed = tmp_path / "same", tmp_path / "changed"
    _tree(str(same))
    _tree(str(changed), alter="mixture_experts_layer_scores_b300/csrc/grouped_swiglu.cu")
    monkeypatch.setattr(bench, "ROOT", str(same))
    gather, copy = bench.recorded_traffic(C["handbook"], True), bench.recorded_traffic(C["handbook"], False)
    assert (gather, copy) == (1400000000, 1500000000)
    assert bench.recorded_traffic(C["mixtral"], False) is None  # no record for that workload
    monkeypatch.setattr(bench, "ROOT", str(changed))
    assert bench.recorded_traffic(C["handbook"], True) is None
    assert bench.recorded_traffic(C["handbook"], False) is None


def test_reference_arm_prints_one_complete_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1", "--config", "tiny"], capture_output=True, text=True, timeout=600,
                         check=True, cwd=ROOT).stdout
    lines = [json.loads(l) for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "tiny" in d["config"]["workload"]


def test_clock_records_that_invalidate_a_number():
    ok = {"sm_mhz": 1432.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}
    assert bench.clock_problem(ok) is None
    assert bench.clock_problem({"sm_mhz": 2000.0, "sm_max_mhz": 2032.0, "reasons": []}) is None
    assert "hw_thermal_slowdown" in bench.clock_problem(dict(ok, reasons=["hw_thermal_slowdown", "sw_power_cap"]))
    assert "sw_thermal_slowdown" in bench.clock_problem(dict(ok, reasons=["sw_thermal_slowdown"]))
    assert "no reason" in bench.clock_problem({"sm_mhz": 900.0, "sm_max_mhz": 2032.0, "reasons": []})
    assert bench.clock_problem({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}) is None


def test_clock_summary_keeps_the_timed_window(tmp_path):
    """nvidia-smi rows are parsed and only those inside the timed region's host-time window
    are summarised (or the nearest few when the region is shorter than the sampling period)."""
    import datetime
    rows = []
    t0 = datetime.datetime(2026, 12, 3, 6, 0, 0)
    for i, (mhz, pw, cap) in enumerate([(2032, 300, "Not Active"), (1500, 1090, "Active"), (1400, 1100, "Active"),
                                        (2032, 250, "Not Active")]):
        ts = (t0 + datetime.timedelta(milliseconds=100 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        rows.append(f"{ts}, 0, {mhz}, 2032, {pw}, 0x0, Not Active, Not Active, Not Active, {cap}")
    s = bench.ClockSampler(0)
    s.proc = object()
    s.path = str(tmp_path / "clk.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    w0 = t0.timestamp()
    d = s.summary((w0 + 0.05, w0 + 0.25))
    assert d["samples"] == 2 and d["sm_mhz"] == 1450 and d["reasons"] == ["sw_power_cap"]
    assert d["power_w_max"] == 1100 and d["scope"] == "timed region"
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    d = s.summary((w0 + 0.101, w0 + 0.102))
    assert d["scope"].startswith("nearest") and d["samples"] == 3


def test_router_bound_takes_the_slower_of_bytes_and_split_products():
    """The router's roofline time: DeepSeek-V3 shape on tensor cores is bound by its three
    bf16 products per weight (3 * 2 N D E flops), the fp32 CUDA-core router by its bytes."""
    pk = {"hbm_gbs": 6425.0, "bf16_tflops": 1808.6}
    cfg = synth.CONFIGS["deepseek_v3"]
    alg = bench.algorithmic(cfg)
    r = bench.router_bound(alg, 100.0, pk, True)
    t_flops = 3 * 2.0 * cfg.N * cfg.D * cfg.E / 1808.6e12
    assert r["bound"] == "tensor" and abs(r["bound_us"] - t_flops * 1e6) < 0.01
    assert abs(r["bound_time_frac"] - t_flops / 100e-6) < 1e-9
    tiny = synth.CONFIGS["tiny"]
    a2 = bench.algorithmic(tiny)
    r2 = bench.router_bound(a2, 10.0, pk, False)
    t_bytes = a2["router_bytes"] / 6425e9
    assert r2["bound"] == "hbm" and abs(r2["bound_us"] - round(t_bytes * 1e6, 2)) < 1e-9
