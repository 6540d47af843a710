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
    assert len(set(base.values())) == len(base)

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
    for k in ("moe_decode_stack", "tc_gemm"):
        e = d[k]
        assert len(e["src_digest"]) == 16 and int(e["src_digest"], 16) >= 0
        # reported while the sources match the capture, else null (never a stale figure)
        want = float(e["dram_bytes_per_unit"]) if e["src_digest"] == bench._src_digest(k) else None
        assert bench._traffic(k, 1.0) == want
    # the decode stack moves its algorithmic bytes and little more (no re-reads)
    alg = 48 * (10 * 811008 + 512 * 2048 * 4 + 2 * 2048 * 4)
    assert 1.0 <= d["moe_decode_stack"]["dram_bytes_per_unit"] / alg < 1.01
