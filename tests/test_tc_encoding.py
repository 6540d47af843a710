"""The tcgen05 descriptor encoders against the documented sm_100 bit layout (values worked out
by hand below), compiled as host code with nvcc: no GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_moe_expert_rl_gb300", "csrc")


@pytest.fixture(scope="module")
def encoded(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("tc")
    src = d / "enc.cu"
    src.write_text('#define RL_TC_HOST_ONLY\n#include <cstdio>\n#include "tc_desc.cuh"\n'
                   "int main(){\n"
                   ' printf("%llx\\n", (unsigned long long)rl::tc::smem_desc(0x12340u, 128u, 1024u));\n'
                   ' printf("%llx\\n", (unsigned long long)rl::tc::smem_desc(0x3fff0u, 2048u, 16u));\n'
                   ' printf("%x\\n", rl::tc::instr_desc(1u, 128, 16));\n'
                   ' printf("%x\\n", rl::tc::instr_desc(0u, 128, 128));\n'
                   ' printf("%x\\n", rl::tc::instr_desc(1u, 64, 256));\n'
                   ' printf("%llx\\n", (unsigned long long)rl::tc::smem_desc_sw128(0x21000u, 1024u));\n'
                   " return 0;}\n")
    exe = d / "enc"
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()


def test_smem_descriptor(encoded):
    # start 0x12340 >> 4 = 0x1234 in bits 0-13; LBO 128 >> 4 = 8 at bit 16; SBO 1024 >> 4 = 64
    # at bit 32; version 1 at bit 46; no swizzle (bits 61-63 = 0)
    assert int(encoded[0], 16) == 0x1234 | (8 << 16) | (64 << 32) | (1 << 46) == 0x0000404000081234
    # start 0x3fff0 >> 4 = 0x3fff (14 bits full); LBO 2048 >> 4 = 128; SBO 16 >> 4 = 1
    assert int(encoded[1], 16) == 0x3FFF | (128 << 16) | (1 << 32) | (1 << 46)


def test_instruction_descriptor(encoded):
    # D f32 (1 << 4); A, B bf16 (1 << 7, 1 << 10); N = 16 -> 2 << 17; M = 128 -> 8 << 24
    assert int(encoded[2], 16) == 0x08040490
    # f16 operands: format 0; N = 128 -> 16 << 17; M = 128
    assert int(encoded[3], 16) == 0x08200010
    # M = 64 -> 4 << 24; N = 256 -> 32 << 17
    assert int(encoded[4], 16) == (1 << 4) | (1 << 7) | (1 << 10) | (32 << 17) | (4 << 24)


def test_swizzled_descriptor(encoded):
    # 128-byte swizzle, K-major: start 0x21000 >> 4 = 0x2100; LBO field 1 (unused with this
    # layout); SBO 1024 >> 4 = 64 at bit 32; version 1 at bit 46; layout 2 in bits 61-63
    assert int(encoded[5], 16) == 0x2100 | (1 << 16) | (64 << 32) | (1 << 46) | (2 << 61)
