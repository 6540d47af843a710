"""Oracle pins for the router: closed forms, brute-force selection on tiny inputs, the tie rule
(including -0.0 against +0.0), the renormalised weights, lookup/miss/flag and slot-order
invariance."""
import itertools
import math

import numpy as np

import oracle
from oracle import NO_EARLY_OUT


def _select_by_repeated_max(row, k):
    """Independent selection: k times, take the largest remaining value, lowest index on ties.
    Values are compared with Python floats, for which -0.0 == +0.0."""
    left = list(range(len(row)))
    out = []
    for _ in range(k):
        best = left[0]
        for e in left[1:]:
            if float(row[e]) > float(row[best]):
                best = e
        out.append(best)
        left.remove(best)
    return out


def test_logits_closed_form_one_hot_rows():
    rng = np.random.default_rng(0)
    H, E = 64, 8
    x = rng.standard_normal((3, H))
    W = np.zeros((E, H))
    cols = rng.integers(0, H, E)
    c = rng.uniform(-2, 2, E)
    W[np.arange(E), cols] = c
    lg = oracle.router_logits(x, W)
    assert np.array_equal(lg, x[:, cols] * c[None, :])


def test_logits_against_sequential_sum():
    rng = np.random.default_rng(1)
    H, E = 48, 5
    x = rng.standard_normal((2, H))
    W = rng.standard_normal((E, H))
    b = rng.standard_normal(E)
    lg = oracle.router_logits(x, W, b)
    for t in range(2):
        for e in range(E):
            acc = math.fsum(float(W[e, h]) * float(x[t, h]) for h in range(H)) + float(b[e])
            assert abs(lg[t, e] - acc) <= 1e-13 * (1 + abs(acc))


def test_topk_all_permutations_distinct():
    for E in range(1, 7):
        for perm in itertools.permutations(range(E)):
            row = np.array(perm, dtype=np.float32) - 2.5
            for k in range(1, E + 1):
                assert oracle.select_topk(row[None, :], k)[0].tolist() == _select_by_repeated_max(row, k)


def test_topk_every_tie_pattern():
    vals = [-1.0, 0.0, 1.0]
    E = 6
    for pat in itertools.product(vals, repeat=E):
        row = np.array(pat, dtype=np.float32)
        for k in (1, 3, 6):
            assert oracle.select_topk(row[None, :], k)[0].tolist() == _select_by_repeated_max(row, k)


def test_signed_zero_is_a_tie():
    for row in ([-0.0, 0.0, -1.0], [0.0, -0.0, -1.0], [-1.0, -0.0, 0.0], [-1.0, 0.0, -0.0]):
        r = np.array(row, dtype=np.float32)
        ids = oracle.select_topk(r[None, :], 3)[0].tolist()
        zeros = [i for i, v in enumerate(row) if v == 0.0]
        assert ids[:2] == zeros and ids[2] not in zeros


def test_weights_invariants():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((50, 32)) * 3
    ids = oracle.select_topk(lg, 8)
    w = oracle.renorm_weights(lg, ids)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)                 # descending logits -> descending weights
    # K equal logits -> 1/K each
    eq = np.full((1, 10), 0.75)
    assert np.allclose(oracle.renorm_weights(eq, oracle.select_topk(eq, 4)), 0.25, rtol=0, atol=1e-15)
    # K = 2 closed form: w0 = 1 / (1 + exp(l1 - l0))
    two = np.array([[0.3, 1.9, -4.0]])
    w2 = oracle.renorm_weights(two, oracle.select_topk(two, 2))
    assert abs(w2[0, 0] - 1.0 / (1.0 + math.exp(0.3 - 1.9))) < 1e-15
    # one dominant logit -> w0 -> 1
    dom = np.array([[50.0, 0.0, 0.1, -0.2]])
    wd = oracle.renorm_weights(dom, oracle.select_topk(dom, 3))[0]
    assert wd[0] == 1.0 - (wd[1] + wd[2]) or abs(wd[0] - 1.0) <= 2e-16
    assert wd[1] < 1e-21 and wd[2] < 1e-21


def test_lookup_miss_and_flag_bruteforce():
    rng = np.random.default_rng(3)
    E, T, K = 16, 7, 4
    table = rng.integers(1, 2 ** 40, E).astype(np.uint64) * np.uint64(16)
    table[rng.choice(E, 5, replace=False)] = 0
    lg = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.route_from_logits(lg, table, K, layer=9, early_out=NO_EARLY_OUT)
    brute_miss = sum(1 for t in range(T) for k in range(K) if table[r.ids[t, k]] == 0)
    assert r.miss == brute_miss
    for t in range(T):
        for k in range(K):
            assert r.slots[t, k] == table[r.ids[t, k]]
    assert r.early_out == (9 if brute_miss else NO_EARLY_OUT)
    # flag keeps the earliest layer
    assert oracle.route_from_logits(lg, table, K, 9, early_out=4).early_out == 4
    # all resident -> no miss, flag untouched; nothing resident -> T*K misses
    full = np.arange(1, E + 1, dtype=np.uint64) * np.uint64(16)
    r2 = oracle.route_from_logits(lg, full, K, 3)
    assert r2.miss == 0 and r2.early_out == NO_EARLY_OUT
    r3 = oracle.route_from_logits(lg, np.zeros(E, np.uint64), K, 3)
    assert r3.miss == T * K and r3.early_out == 3


def test_route_decides_on_f32_logits():
    """Two logits that differ in f64 but round to the same f32 value are a tie (lower index)."""
    H, E = 4, 3
    W = np.zeros((E, H))
    W[0, 0] = 1.0
    W[1, 0] = 1.0 + 2.0 ** -40          # larger in f64, equal after rounding to f32
    W[2, 0] = 0.5
    xn = np.array([[1.0, 0, 0, 0]])
    table = np.arange(1, E + 1, dtype=np.uint64)
    r = oracle.route(xn, W, None, table, 2, 0)
    assert r.ids[0].tolist() == [0, 1]
