"""Host-side bookkeeping of bench.py: the DRAM traffic recorded from an ncu capture counts only
while the profiled kernel's translation unit (its .cu file and the headers it includes) is
unchanged apart from comments, and each kernel's digest ignores the other kernels' files."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path):
    for d in ("include", os.path.join("quantized_moe_expert_rl_gb300", "csrc")):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d)
    return str(tmp_path), tmp_path / "quantized_moe_expert_rl_gb300" / "csrc"


def test_digest_follows_the_translation_unit(tmp_path):
    root, csrc = _tree(tmp_path)
    base = {k: bench._src_digest(k, root) for k in bench._KERNEL_TU}
    assert base == {k: bench._src_digest(k) for k in bench._KERNEL_TU}
    # one digest per translation unit: kernels built from the same unit share it
    assert len(set(base.values())) == len(set(bench._KERNEL_TU.values()))
    assert base["moe_decode_layer"] == base["moe_decode_stack"]

    # a comment-only change keeps every digest
    p = csrc / "stack_kernel.cuh"
    p.write_text(p.read_text() + "\n// a comment\n/* and a block\n comment */\n")
    assert {k: bench._src_digest(k, root) for k in bench._KERNEL_TU} == base

    # a code change in a header of the stack kernel changes its digest only
    p.write_text(p.read_text() + "\nstatic const int probe_value = 1;\n")
    now = {k: bench._src_digest(k, root) for k in bench._KERNEL_TU}
    assert now["moe_decode_stack"] != base["moe_decode_stack"]
    assert now["tc_gemm"] == base["tc_gemm"] and now["moe_decode"] == base["moe_decode"]

    # a header every kernel includes changes them all
    p = csrc / "rl_common.cuh"
    p.write_text(p.read_text() + "\nstatic const int probe_value2 = 2;\n")
    now2 = {k: bench._src_digest(k, root) for k in bench._KERNEL_TU}
    assert all(now2[k] != now[k] for k in bench._KERNEL_TU)


def test_recorded_traffic_is_per_launch():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for k in ("moe_decode_stack", "moe_decode_layer", "tc_gemm"):
        e = d[k]
        assert len(e["src_digest"]) == 16 and int(e["src_digest"], 16) >= 0
        # reported while the sources match the capture, else null (never a stale figure)
        want = float(e["dram_bytes_per_unit"]) if e["src_digest"] == bench._src_digest(k) else None
        assert bench._traffic(k, 1.0) == want
    # the decode stack reads its algorithmic bytes and little more (no re-reads); the writes
    # of a capture include dirty L2 lines that earlier launches left behind
    alg = 48 * (10 * 811008 + 512 * 2048 * 4 + 2 * 2048 * 4)
    e = d["moe_decode_stack"]
    assert 1.0 <= e["dram_bytes_read_per_unit"] / alg < 1.01
    assert e["dram_bytes_read_per_unit"] <= e["dram_bytes_per_unit"] < 1.02 * alg


def test_clock_summary_reads_reasons_and_median():
    """nvidia-smi lines (index, clocks.sm, clocks.max.sm, power, active mask, hw_slowdown,
    hw_thermal, sw_thermal, sw_power_cap) -> median SM clock, max clock, active reasons."""
    c = bench.ClockSampler(0)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1900, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2055, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage line", ""]
    s = c.summary()
    assert s == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = ["0, 1200, 2070, 700.0, 0x8, Active, Not Active, Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]


def test_reference_arm_prints_one_contract_line():
    """--impl reference on CPU: one JSON line with the keys of the bench contract, the oracle
    timed on this host's cores over a bounded sample."""
    import subprocess
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-step-s", "0.5"], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "decode_stack" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    st = d["cpu_baseline"]["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] - 1000.0 * d["config"]["tokens_per_step"] / d["value"]) < 1e-6 * d["ms_per_step"]
