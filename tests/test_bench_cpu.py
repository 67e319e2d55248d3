"""bench.py's contract on the CPU: the reference arm (the oracle on the host
cores) prints one JSON line with the fields the measurement contract names,
and the warm-up floor is enforced."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def _bench(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--workload", "square256", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["M"] == d["config"]["N"] == d["config"]["K"] == 256


def test_warmup_floor():
    r = _bench("--impl", "reference", "--workload", "square256", "--steps", "3", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_clocks_summary_prefers_samples_inside_the_region():
    """NVML samples from inside the timed region decide the clocks entry; the
    reason bits decode to nvidia-smi's names; without samples the nvidia-smi
    summary stands."""
    sys.path.insert(0, ROOT)
    import bench
    smi = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3, "note": "nearest samples"}
    assert bench.clocks_summary([], smi) == smi
    rows = [(2070.0, 2070.0, 0x0), (1980.0, 2070.0, 0x4), (2070.0, 2070.0, 0x1), (1500.0, 2070.0, 0x8 | 0x40)]
    c = bench.clocks_summary(rows, smi)
    assert c["sm_mhz"] == 2025.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] == 4
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert c["nvidia_smi"] == smi


def test_source_hash_ignores_comments_only():
    """The hash that ties a recorded DRAM count to the code changes with the
    code, not with its comments."""
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {\n    return x + 1;   // one more\n}\n/* note */\n"
    b = "int f(int x) {\n    return x + 1;   // one more, reworded\n}\n/* another\n   note */\n"
    c = "int f(int x) {\n    return x + 2;   // one more\n}\n/* note */\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    # a comment grown by a line, or code re-wrapped, leaves the code as it was
    d = "int f(int x) {\n    // one\n    // more\n    return x +\n        1;\n}\n"
    assert bench._code_only(a) == bench._code_only(d)


def test_profiler_style_shape_flags():
    """--m --n --k (with --A --B --C --split-k --persistent) time an ad-hoc GEMM;
    the reference arm takes the same flags and labels the line with them."""
    r = _bench("--impl", "reference", "--m", "64", "--n", "48", "--k", "40", "--A", "col", "--B", "row",
               "--C", "f32", "--split-k", "2", "--persistent", "0", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    c = d["config"]
    assert (c["M"], c["N"], c["K"], c["out"], c["split_k"]) == (64, 48, 40, "f32", 2)
    assert c["layout_a"] == "column-major" and c["layout_b"] == "row-major"
    assert c["launch"] == "one cluster per tile"
    r = _bench("--impl", "reference", "--m", "64", "--steps", "3", "--warmup", "3", timeout=120)
    assert r.returncode != 0 and "--m, --n and --k go together" in r.stderr


def test_both_arms_label_a_workload_alike():
    """The reference arm's data and config come from the same builders as the
    GPU arm's, so the two lines name the same workload."""
    sys.path.insert(0, ROOT)
    import bench
    w = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert bench.DEFAULT_WORKLOAD == "large" and (w["M"], w["N"], w["K"]) == (16384, 8192, 8192)
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert src.count('"config": workload_config(w)') == 2
    assert src.count('"data": workload_data(w, seed)') == 2
    assert src.count('"config": conv_config(w)') == 2


def test_conv_labels_agree_with_the_library():
    """The conv line's P, Q (the reference arm computes them without a GPU)
    agree with the library's own gemm_conv2d_out_dims for every benched
    convolution."""
    sys.path.insert(0, ROOT)
    import bench
    import dense_tensor_core_bf16_gb300 as g
    for name, w in bench.WORKLOADS.items():
        cv = w.get("conv")
        if not cv:
            continue
        d = g.gemm_conv2d_desc_t(N=cv["N"], H=cv["H"], W=cv["W"], C=cv["C"], K=cv["K"], R=cv["R"], S=cv["S"],
                                 pad_h=cv["pad"][0], pad_w=cv["pad"][1], stride_h=cv["stride"][0],
                                 stride_w=cv["stride"][1], dil_h=cv["dil"][0], dil_w=cv["dil"][1])
        st, P, Q = g.gemm_conv2d_out_dims(d)
        assert st == 0 and (P, Q) == bench.conv_out_dims(cv), name
        c = bench.conv_config(w)
        assert c["gemm"] == {"M": cv["N"] * P * Q, "N": cv["K"], "K": cv["R"] * cv["S"] * cv["C"]}


def test_custom_workload_descriptor():
    sys.path.insert(0, ROOT)
    import bench
    w = bench.custom_workload(300, 520, 264, "col", "row", "f32", 3, 0, "int4")
    assert (w["M"], w["N"], w["K"], w["out"], w["split_k"]) == (300, 520, 264, "f32", 3)
    assert w["a_col"] and w["b_row"] and w["non_persistent"] and not w["scaled"]
    c = bench.workload_config(w)
    assert c["layout_a"] == "column-major" and c["layout_b"] == "row-major" and c["launch"] == "one cluster per tile"
