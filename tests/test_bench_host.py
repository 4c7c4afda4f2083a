"""Host-side logic of bench.py: the profile-to-code binding of the ncu
traffic figure, the clock summary, and the JSON line of the reference arm
(the CPU oracle), which needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_text_ignores_comments_and_whitespace():
    a = "int f(int x) {  // twice\n  return 2 * x; /* doubled */\n}\n"
    b = "/* header\n   comment */\nint f(int x) {\n\treturn 2 * x;\n}"
    c = "int f(int x) { return 3 * x; }"
    assert bench.code_text(a) == bench.code_text(b) == "int f(int x) { return 2 * x; }"
    assert bench.code_text(c) != bench.code_text(a)


def test_profiled_traffic_is_bound_to_the_kernel_code(tmp_path):
    h = bench.source_hash()
    good = tmp_path / "good.md"
    good.write_text(f"x\ndram_bytes_per_launch: 123456\nkernel_code_sha256: {h}\n")
    stale = tmp_path / "stale.md"
    stale.write_text("dram_bytes_per_launch: 123456\nkernel_code_sha256: " + "0" * 64 + "\n")
    partial = tmp_path / "partial.md"
    partial.write_text(f"kernel_code_sha256: {h}\n")
    assert bench.profiled_traffic(str(good)) == 123456
    assert bench.profiled_traffic(str(stale)) is None
    assert bench.profiled_traffic(str(partial)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None


def test_committed_profile_parses():
    """The committed fprop summary carries both keys the bench reads."""
    text = open(os.path.join(ROOT, "profiles", "k_gemm_nvfp4_fprop_ultra.md")).read()
    assert "dram_bytes_per_launch:" in text and "kernel_code_sha256:" in text


def test_summarise_clocks():
    rows = [
        "1920, 2032, 1050.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "1905, 2032, 1099.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "[N/A], 2032, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1890, 2032, [N/A], 0x0000000000000008, Active, Not Active, Not Active, Not Active",
    ]
    s = bench.summarise_clocks("\n".join(rows))
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1905 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["power_w_max"] == 1099.0
    assert bench.summarise_clocks("") is None
    assert bench.summarise_clocks("a, b, c\n") is None


def test_workload_config_names_the_workload():
    from nvfp4_precision_02_b300 import workloads as wl
    m = wl.ULTRA_MOE
    c = bench.workload_config("ultra", wl.ULTRA_DENSE, m, m.tokens * m.topk, 2)
    assert c["workload"] == "ultra_full_step" and c["moe_rows"] == 360448
    assert c["in_proj_out"] == 33024 and c["parallelism"] == "replicas x2"
    assert "model" not in c


def _run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_json_line():
    """`--impl reference` times the oracle on the host and prints one JSON
    line with the contract's keys; value, cpu_baseline and e2e agree."""
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "super"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "super_full_step"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""



def test_gemm_roofline_and_bytes_table():
    from nvfp4_precision_02_b300 import workloads as wl
    d, m = wl.ULTRA_DENSE, wl.ULTRA_MOE
    R = m.tokens * m.topk
    tab = bench.gemm_bytes_table(d, m, R)
    src = open(os.path.join(ROOT, "bench.py")).read()
    ops_src = src[src.index("self.ops = ["):src.index("self.gemm_flops")]
    for name in tab:                       # every key names a GEMM op of the step
        assert f'("{name}", "tensor"' in ops_src, name
    # fprop: (16384 + 33024) x 8192 FP4 operands and a bf16 16384 x 33024 output
    assert tab["gemm fprop"] == 0.5625 * (16384 + 33024) * 8192 + 2 * 16384 * 33024
    # up-projection: all 512 experts' 5120 x 2048 weights are read once
    assert tab["grouped_gemm up (+ per-expert amax of H)"] == 0.5625 * (360448 + 512 * 5120) * 2048 + 2 * 360448 * 5120
    # 1 GB at 1000 GB/s is 1 ms; 2 TFLOP at 1000 TFLOP/s is 2 ms: tensor-bound, 2 ms roof
    r = bench.gemm_roofline(2e12, 1e9, 4.0, 1000.0, 1000.0)
    assert r["bound"] == "tensor" and r["roofline_ms"] == 2.0 and r["frac_roofline"] == 0.5
    r = bench.gemm_roofline(0.5e12, 1e9, 2.0, 1000.0, 1000.0)
    assert r["bound"] == "hbm" and r["roofline_ms"] == 1.0 and r["frac_roofline"] == 0.5
    assert bench.gemm_roofline(1e12, None, 1.0, 1.0, 1.0) == {}
    # with the measured peaks the dense GEMMs are tensor-bound and the up-projection HBM-bound
    hbm, fp4 = 6487.7, 1377.6 * 6
    flops = 2.0 * 16384 * 33024 * 8192
    assert bench.gemm_roofline(flops, tab["gemm fprop"], 1.7, hbm, fp4)["bound"] == "tensor"
    up = 2.0 * R * m.expert_hidden * m.latent
    assert bench.gemm_roofline(up, tab["grouped_gemm up (+ per-expert amax of H)"], 2.4, hbm, fp4)["bound"] == "hbm"



def test_alu_roofline():
    # 541 M elements x ops at 64 lanes x 148 SMs x 2032 MHz
    r = bench.alu_roofline(16384 * 33024, 0.95, 2032.0, 148)
    n = bench.SR_ALU_OPS_PER_ELEMENT
    assert r["bound"] == "alu" and r["ops_per_element"] == n
    assert abs(r["floor_ms"] - 16384 * 33024 * n / (64 * 148 * 2032e6) * 1e3) < 1e-4
    assert abs(r["frac"] - r["floor_ms"] / 0.95) < 1e-3
    assert bench.alu_roofline(100, 1.0, None, 148) is None


def test_fp4_peaks_and_fractions():
    pk = {"hbm_gbs": 6500.0, "bf16_burst": 1700.0, "bf16_sustained": 1300.0, "source": "measured"}
    fp4 = bench.fp4_peaks(pk, 148, 2000.0)
    assert fp4["burst_x6"] == 10200.0 and fp4["sustained_x6"] == 7800.0 and fp4["datasheet"] == 13500.0
    # 32768 (measured MMA issue) and 49152 (counter) FLOP per SM per clock x 148 SMs x 2 GHz
    assert abs(fp4["mma_issue_at_clock"] - 32768 * 148 * 2.0e9 / 1e12) < 1e-6
    assert abs(fp4["counter_at_clock"] - 49152 * 148 * 2.0e9 / 1e12) < 1e-6
    assert "mma_issue_at_clock" not in bench.fp4_peaks(pk, 148, None)
    f = bench.gemm_fracs(5100.0, fp4)
    assert f["frac_fp4_burst_x6"] == 0.5 and f["frac_fp4_datasheet"] == round(5100 / 13500, 4)
    e = bench.op_entry("hbm", 6.5e9, 1.0, pk, fp4)      # 6.5 GB in 1 ms
    assert e["gbs"] == 6500.0 and e["frac_hbm"] == 1.0 and e["frac_hbm_nominal_8tbs"] == round(6500 / 8000, 4)
    g = bench.op_entry("tensor", 10.2e12, 1.0, pk, fp4, nbytes=1e9)
    assert g["tflops"] == 10200.0 and g["frac_fp4_burst_x6"] == 1.0 and g["bound"] == "tensor"


def test_config_ops_cover_the_step():
    """c2-c4 partition the step's ops: fprop, backward, LatentMoE."""
    src = open(os.path.join(ROOT, "bench.py")).read()
    ops_src = src[src.index("self.ops = ["):src.index("self.gemm_flops")]
    names = [l.split('"')[1] for l in ops_src.splitlines() if l.strip().startswith('("')]
    spans = sorted(bench.CONFIG_OPS.values())
    assert spans[0][0] == 0 and spans[-1][1] == len(names)
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    c2, c3, c4 = (names[i0:i1] for i0, i1 in (bench.CONFIG_OPS[k] for k in ("c2", "c3", "c4")))
    assert c2[-1] == "gemm fprop" and "gemm dgrad" in c3 and "gemm wgrad" in c3
    assert c4[-1] == "grouped_gemm down"


def test_gpus_n_starts_n_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself
    (torch.distributed.run on 127.0.0.1); the launch check joins them with
    gloo on CPU and rank 0 reports n_gpus = 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--launch-check"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["world_size"] == 2


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))


# Kernels of the Ultra step's launch list (profiles/launches_ultra_full_step.md)
# and the ncu summaries that cover them, with the sources each summary's
# kernel_code_sha256 is taken over.
_Q = "nvfp4_precision_02_b300/csrc/"
STEP_KERNEL_SUMMARIES = {
    "k_gemm_nvfp4<bf16, TMA store, pair, groups along M>": ["k_gemm_nvfp4_grouped_up_super.md",
                                                            "k_gemm_nvfp4_grouped_down_super.md"],
    "k_gemm_nvfp4<bf16, TMA store, pair, dense>": ["k_gemm_nvfp4_fprop_ultra.md", "k_gemm_nvfp4_dgrad_ultra.md"],
    "k_gemm_nvfp4<fp32, TMA store, pair, dense>": ["k_gemm_nvfp4_wgrad_ultra.md"],
    "k_quant2d_w<2>": ["k_quant2d_w_moe_super.md"],
    "k_amax": ["k_amax_ultra.md"],
    "k_quant1d<RNE, grouped, band>": ["k_quant1d_grouped_h_ultra.md"],
    "k_rht<4>": ["k_rht_dual_sr_ultra.md"],
    "k_amax_grouped": ["k_amax_grouped_super.md"],
    "k_rht_stream<3>": ["k_rht_stream_dual_amax_ultra.md"],
    "k_quant2d": ["k_quant2d_ultra.md"],
    "k_rht_stream<1>": ["k_rht_stream_rne_ultra.md"],
    "k_quant1d<RNE>": ["k_quant1d_rne_ultra.md"],
    "k_rht_stream<0>": ["k_rht_stream_amax_ultra.md"],
}


def _summary_sources(name):
    if name.startswith("k_gemm"):
        return bench.GEMM_SOURCES
    if name.startswith("k_quant2d_w"):
        return (_Q + "quant2d_w.cuh",) + bench.QUANT_SOURCES
    if name.startswith("k_quant2d_resident"):
        return (_Q + "quant2d_resident.cuh",) + bench.QUANT_SOURCES
    return bench.QUANT_SOURCES


def test_every_step_kernel_has_an_ncu_summary():
    """Each kernel in the step's launch list has a committed ncu summary with
    its DRAM bytes and code hash; a summary whose hash no longer matches its
    sources is reported (the kernel changed after the capture)."""
    import re
    import warnings
    with open(os.path.join(ROOT, "profiles", "launches_ultra_full_step.md")) as f:
        text = f.read()
    labels = [m.group(1).strip() for m in re.finditer(r"^\| (k_[^|(]+?)\s*(?:\([^|]*\))? \| \d+ \|", text, re.M)]
    assert labels, "no kernel rows in the launch list"
    for lab in labels:
        assert lab in STEP_KERNEL_SUMMARIES, f"launch-list kernel without a summary: {lab}"
        for name in STEP_KERNEL_SUMMARIES[lab]:
            with open(os.path.join(ROOT, "profiles", name)) as f:
                body = f.read()
            assert re.search(r"dram_bytes_per_launch:\s*\d+", body), name
            h = re.search(r"kernel_code_sha256:\s*([0-9a-f]{64})", body)
            assert h, name
            if h.group(1) != bench.source_hash(_summary_sources(name)):
                warnings.warn(f"{name}: kernel code changed since the capture")
