"""The seeded input generator: pinned to the published SplitMix64 sequence, IEEE binary16
rounding, and plain properties of the distributions it is asked to draw."""
import math

import numpy as np

import synth


def test_splitmix64_published_sequence():
    # The first outputs of SplitMix64 seeded with 1234567, as published with the reference
    # implementation (Vigna, splitmix64.c) and reproduced by many test suites.
    expected = [6457827717110365317, 3203168211198807973, 9817491932198370423,
                4593380528125082431, 16408922859458223821]
    assert [synth.lib().synth_draw(1234567, i) for i in range(5)] == expected


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(1e-3, 4e-3, 20000), rng.uniform(-70000, 70000, 2000),
                           rng.uniform(-1e-6, 1e-6, 2000), [0.0, -0.0, 65504.0, 6.103515625e-05]])
    ours = np.array([synth.lib().synth_f16_bits(float(v)) for v in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_ln_and_sincos_accuracy():
    L = synth.lib()
    for u in [2.0 ** -53, 1e-300, 1e-10, 0.1, 0.5, 0.7071, 0.99999, 1.0, 2.5, 1e10]:
        assert abs(L.synth_ln(u) - math.log(u)) <= 4e-16 * max(1.0, abs(math.log(u)))
    import ctypes
    s, c = ctypes.c_double(), ctypes.c_double()
    for v in np.linspace(0, 1, 1001, endpoint=False):
        L.synth_sincos2pi(float(v), ctypes.byref(s), ctypes.byref(c))
        assert abs(s.value - math.sin(2 * math.pi * v)) < 2e-15
        assert abs(c.value - math.cos(2 * math.pi * v)) < 2e-15


def test_grid_and_blocks():
    g = synth.grid(0)
    assert g.shape == (256, 8) and set(np.unique(g)) == {8, 25, 43}
    counts = np.bincount(g.reshape(-1).astype(np.int64))[[8, 25, 43]]
    assert np.all(np.abs(counts - 2048 / 3) < 100)
    blk = synth.matrix_blocks(0, 3, 1, 64).reshape(64, 66)
    d = (blk[:, 0].astype(np.uint16) | (blk[:, 1].astype(np.uint16) << 8)).view(np.float16)
    assert np.all((d >= np.float16(1e-3)) & (d <= np.float16(4e-3)))
    assert np.array_equal(blk.reshape(-1), synth.matrix_blocks(0, 3, 1, 64))       # deterministic
    assert not np.array_equal(blk.reshape(-1), synth.matrix_blocks(0, 3, 2, 64))   # keyed by matrix


def test_normals_and_records():
    w = synth.WORKLOADS["decode_layer"]
    wr = synth.router(w, 0)
    assert wr.shape == (512, 2048) and abs(wr.std() - 0.02) < 3e-4 and abs(wr.mean()) < 3e-4
    x = synth.tokens(w, 0, 8)
    assert abs(x.std() - 1.0) < 0.03
    rec = synth.expert_records(w, 5, 7, 2)
    assert rec.shape == (2, 811008)
    # record = [gate | up | down] = matrices 0, 1, 2 of that expert
    mb = w.matrix_bytes
    assert np.array_equal(rec[1, mb:2 * mb], synth.matrix_blocks(5, 8, 1, mb // 66))


def test_zipf_and_residency():
    w = synth.WORKLOADS["prefill_bounded"]
    b = synth.zipf_bias(w, 3)
    ranks = np.rint(np.exp(-b.astype(np.float64) / 1.1)).astype(np.int64)
    assert sorted(ranks.tolist()) == list(range(1, 513))
    m = synth.resident_mask(w, 3)
    assert m.sum() == 435 and set(np.unique(m)) == {0, 1}
    assert not np.array_equal(m, synth.resident_mask(w, 4))
