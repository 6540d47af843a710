"""Oracle pins for the block format: hand-built blocks, IEEE binary16, brute-force round trip,
the flat layout of 128-value rows."""
import os

import numpy as np
import pytest

import oracle


def _load_golden(golden_dir):
    grid = np.full((256, 8), 8, dtype=np.int8)
    blocks, expects = {}, []
    with open(os.path.join(golden_dir, "blocks_handbuilt.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "grid":
                grid[int(tok[1])] = [int(v) for v in tok[2:10]]
            elif tok[0] == "block":
                blocks[tok[1]] = np.frombuffer(bytes.fromhex(tok[2]), dtype=np.uint8)
            elif tok[0] == "expect":
                expects.append((tok[1], int(tok[2]), [float(v) for v in tok[3:]]))
    return grid, blocks, expects


def test_handbuilt_blocks(golden_dir):
    grid, blocks, expects = _load_golden(golden_dir)
    assert all(b.size == 66 for b in blocks.values())
    decoded = {k: oracle.dequantize(v, 256, grid) for k, v in blocks.items()}
    for name, first, vals in expects:
        got = decoded[name][first:first + len(vals)]
        assert np.array_equal(got, np.array(vals)), (name, first, got, vals)


def test_fp16_decode_matches_ieee_for_all_finite_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 10) & 0x1F) != 31
    ours = oracle.fp16_to_f64(bits[finite])
    ref = bits[finite].view(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref)
    with pytest.raises(ValueError):
        oracle.fp16_to_f64(np.array([0x7C00], dtype=np.uint16))


def _encode_bruteforce(vals, d_bits, grid):
    """Find (idx, sign) per group whose decoded values equal vals, by trying all 256 x 256."""
    d = float(np.array([d_bits], dtype=np.uint16).view(np.float16)[0])
    out = bytearray([d_bits & 0xFF, d_bits >> 8])
    for g in range(32):
        target = vals[8 * g:8 * g + 8]
        found = None
        for idx in range(256):
            if [abs(d * int(grid[idx][j])) for j in range(8)] != [abs(t) for t in target]:
                continue                                   # magnitudes differ: no sign can match
            for s in range(256):
                cand = [d * int(grid[idx][j]) * (-1 if (s >> j) & 1 else 1) for j in range(8)]
                if cand == list(target):
                    found = (idx, s)
                    break
            if found:
                break
        assert found is not None
        out += bytes(found)
    return np.frombuffer(bytes(out), dtype=np.uint8)


def test_round_trip_bruteforce():
    import synth
    grid = synth.grid(0)
    rng = np.random.default_rng(7)
    d_bits = 0x1C19
    d = float(np.array([d_bits], dtype=np.uint16).view(np.float16)[0])
    rows = rng.integers(0, 256, 32)
    signs = rng.integers(0, 256, 32)
    vals = np.array([d * int(grid[rows[g]][j]) * (-1 if (signs[g] >> j) & 1 else 1)
                     for g in range(32) for j in range(8)])
    enc = _encode_bruteforce(vals, d_bits, grid)
    assert np.array_equal(oracle.dequantize(enc, 256, grid), vals)


def test_flat_layout_of_short_rows():
    """A matrix with 128-value rows is stored flat: row 2b is the first half of block b and
    row 2b+1 the second half."""
    grid = np.zeros((256, 8), dtype=np.int8)
    for i in range(256):
        grid[i] = [i % 43 + 1] * 8
    rows, cols = 4, 128
    blk = bytearray()
    for b in range(2):
        blk += bytes([0x00, 0x3C])                         # d = 1
        for g in range(32):
            blk += bytes([b * 32 + g, 0])                  # idx = global group number
    W = oracle.dequantize(np.frombuffer(bytes(blk), dtype=np.uint8), rows * cols, grid).reshape(rows, cols)
    for r in range(rows):
        for c in range(cols):
            G = (r * cols + c) // 8                        # global group index
            assert W[r, c] == G % 43 + 1


def test_expert_weights_split():
    import synth
    w = synth.WORKLOADS["tiny"]
    grid = synth.grid(0)
    rec = synth.expert_records(w, 0, 3, 1)[0]
    wg, wu, wd = oracle.expert_weights(rec, w.hidden, w.inter, grid)
    assert wg.shape == (128, 512) and wu.shape == (128, 512) and wd.shape == (512, 128)
    mb = w.matrix_bytes
    assert np.array_equal(wd.reshape(-1), oracle.dequantize(rec[2 * mb:], 512 * 128, grid))
    # magnitudes are d * {8, 25, 43} with d in [1e-3, 4e-3]
    a = np.abs(np.concatenate([wg.ravel(), wu.ravel(), wd.ravel()]))
    assert a.min() >= 8 * 1e-3 * (1 - 1e-3) and a.max() <= 43 * 4e-3 * (1 + 1e-3)
