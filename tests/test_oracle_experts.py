"""Oracle pins for the experts, the ordered sum, the pair list, RMSNorm and the stack with
early-out and fill: closed forms, brute force on tiny inputs and invariants."""
import math

import numpy as np

import oracle
import synth
from oracle import NO_EARLY_OUT


def _const_record(hidden, inter, d_bits=0x2000, idx=5, sign=0):
    """Record whose three matrices are all d * grid[idx][j] * sign."""
    nb = hidden * inter // 256
    blk = bytes([d_bits & 0xFF, d_bits >> 8]) + bytes([idx, sign]) * 32
    return np.frombuffer(blk * (3 * nb), dtype=np.uint8)


def test_expert_closed_form_constant_weights():
    H, I = 512, 256
    grid = np.full((256, 8), 8, dtype=np.int8)        # all 8s
    d = 2.0 ** -7                                       # fp16 0x2000
    rec = _const_record(H, I)
    wg, wu, wd = oracle.expert_weights(rec, H, I, grid)
    assert np.all(wg == 8 * d) and np.all(wd == 8 * d)
    x = np.random.default_rng(0).standard_normal(H) * 0.1
    g = 8 * d * x.sum()                                 # every gate/up row gives the same value
    h = g / (1 + math.exp(-g)) * g
    o_expected = 8 * d * I * h                          # every down row sums I equal terms
    o = oracle.expert_forward(wg, wu, wd, x)
    assert np.allclose(o, o_expected, rtol=1e-13, atol=0)


def _decode_bytes_loop(raw, n_values, grid):
    """Independent per-value decoder in plain Python loops."""
    out = []
    for b in range(n_values // 256):
        blk = raw[66 * b: 66 * b + 66]
        bits = int(blk[0]) | (int(blk[1]) << 8)
        e, f = (bits >> 10) & 31, bits & 1023
        dv = (f / 1024) * 2.0 ** -14 if e == 0 else (1 + f / 1024) * 2.0 ** (e - 15)
        dv = -dv if bits >> 15 else dv
        for g in range(32):
            idx, s = int(blk[2 + 2 * g]), int(blk[3 + 2 * g])
            for j in range(8):
                out.append(dv * int(grid[idx][j]) * (-1 if (s >> j) & 1 else 1))
    return out


def test_expert_forward_bruteforce_tiny():
    H, I = 256, 8
    grid = synth.grid(0)
    rng = np.random.default_rng(4)
    nb = H * I // 256
    raw = bytearray()
    for _ in range(3 * nb):
        raw += bytes([rng.integers(0, 256), rng.integers(0x10, 0x20)]) + bytes(rng.integers(0, 256, 64).tolist())
    raw = np.frombuffer(bytes(raw), dtype=np.uint8)
    mb = nb * 66
    Wg = _decode_bytes_loop(raw[:mb], H * I, grid)
    Wu = _decode_bytes_loop(raw[mb:2 * mb], H * I, grid)
    Wd = _decode_bytes_loop(raw[2 * mb:], H * I, grid)
    x = rng.standard_normal(H)
    g = [math.fsum(Wg[i * H + c] * x[c] for c in range(H)) for i in range(I)]
    u = [math.fsum(Wu[i * H + c] * x[c] for c in range(H)) for i in range(I)]
    h = [g[i] / (1 + math.exp(-g[i])) * u[i] for i in range(I)]
    o = [math.fsum(Wd[r * I + i] * h[i] for i in range(I)) for r in range(H)]
    wg, wu, wd = oracle.expert_weights(raw, H, I, grid)
    got = oracle.expert_forward(wg, wu, wd, x)
    assert np.allclose(got, o, rtol=1e-12, atol=1e-12)


def test_ordered_sum_is_a_left_fold():
    # values chosen so that float addition order matters: (1e16 + 1) - 1e16 = 0 but 1 + (1e16 - 1e16) = 1
    outs = np.array([[[1e16], [1.0], [-1e16]]])
    w = np.ones((1, 3))
    assert oracle.ordered_sum(outs, w)[0, 0] == ((1e16 + 1.0) - 1e16)
    outs2 = np.array([[[1.0], [1e16], [-1e16]]])
    assert oracle.ordered_sum(outs2, w)[0, 0] == ((1.0 + 1e16) - 1e16)


def test_k1_and_weights():
    w = synth.WORKLOADS["tiny"]
    grid = synth.grid(0)
    recs = synth.expert_records(w, 0, 0, 2)
    slots = {16: recs[0], 32: recs[1]}
    x = synth.tokens(w, 0, 1).astype(np.float64)
    y = oracle.moe_experts(x, np.array([[0]]), np.array([[1.0]]), np.array([[16]], dtype=np.uint64),
                           slots.__getitem__, w.hidden, w.inter, grid)
    wg, wu, wd = oracle.expert_weights(recs[0], w.hidden, w.inter, grid)
    assert np.array_equal(y[0], oracle.expert_forward(wg, wu, wd, x[0]))
    # two experts: y = w0 o0 + w1 o1
    y2 = oracle.moe_experts(x, np.array([[1, 0]]), np.array([[0.25, 0.75]]),
                            np.array([[32, 16]], dtype=np.uint64), slots.__getitem__, w.hidden, w.inter, grid)
    wg1, wu1, wd1 = oracle.expert_weights(recs[1], w.hidden, w.inter, grid)
    o1 = oracle.expert_forward(wg1, wu1, wd1, x[0])
    assert np.array_equal(y2[0], 0.25 * o1 + 0.75 * oracle.expert_forward(wg, wu, wd, x[0]))


def test_rmsnorm_closed_form():
    for c in (0.5, -3.0, 1e-3):
        x = np.full((1, 2048), c)
        expect = c / math.sqrt(c * c + 1e-6)
        assert np.allclose(oracle.rmsnorm(x), expect, rtol=1e-15, atol=0)
    assert np.allclose(np.sqrt(np.mean(oracle.rmsnorm(np.random.default_rng(1).standard_normal((3, 64)),
                                                      eps=0.0) ** 2, axis=1)), 1.0, rtol=1e-15)


def test_pairs_bruteforce():
    rng = np.random.default_rng(5)
    T, K, E = 37, 4, 12
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    offs, ptok, pk = oracle.build_pairs(ids, E)
    brute = [(t, k) for e in range(E) for t in range(T) for k in range(K) if ids[t, k] == e]
    assert list(zip(ptok.tolist(), pk.tolist())) == brute
    hist = [sum(1 for t in range(T) for k in range(K) if ids[t, k] == e) for e in range(E)]
    assert offs.tolist() == [sum(hist[:e]) for e in range(E + 1)] and offs[-1] == T * K


def test_prefill_equals_per_token_definition():
    w = synth.WORKLOADS["tiny"]
    grid = synth.grid(0)
    recs = synth.expert_records(w, 0, 0, w.n_experts)
    table = (np.arange(w.n_experts, dtype=np.uint64) + 1) * np.uint64(4096)
    source = {int(table[e]): recs[e] for e in range(w.n_experts)}.__getitem__
    x = synth.tokens(w).astype(np.float64)
    r = oracle.route(x, synth.router(w, 0), None, table, w.top_k, 0)
    y_tok = oracle.moe_experts(x, r.ids, r.weights, r.slots, source, w.hidden, w.inter, grid)
    y_pre, pair_out, offs, ptok, pk = oracle.prefill_chunk(x, r.ids, r.weights, r.slots, source,
                                                           w.hidden, w.inter, grid, w.n_experts)
    assert np.array_equal(y_tok, y_pre)


def test_slot_order_invariance():
    """Moving every expert to a different slot address changes nothing but the slot values."""
    w = synth.WORKLOADS["tiny"]
    grid = synth.grid(0)
    recs = synth.expert_records(w, 0, 0, w.n_experts)
    x = synth.tokens(w).astype(np.float64)
    wr = synth.router(w, 0)
    out = []
    for perm in (np.arange(w.n_experts), synth.permutation(synth.TAG_SLOTPERM, 0, w.n_experts)):
        table = (perm.astype(np.uint64) + 1) * np.uint64(811008)   # expert e lives at slot perm[e]
        src = {int(table[e]): recs[e] for e in range(w.n_experts)}.__getitem__
        r = oracle.route(x, wr, None, table, w.top_k, 0)
        y = oracle.moe_experts(x, r.ids, r.weights, r.slots, src, w.hidden, w.inter, grid)
        out.append((r, y, table))
    (r0, y0, t0), (r1, y1, t1) = out
    assert np.array_equal(r0.ids, r1.ids) and np.array_equal(r0.weights, r1.weights)
    assert r0.miss == r1.miss == 0 and np.array_equal(y0, y1)
    assert np.array_equal(r1.slots, t1[r1.ids])


def test_stack_early_out_and_fill():
    w = synth.WORKLOADS["tiny"]
    grid = synth.grid(0)
    L = 4
    recs = {l: synth.expert_records(w, l, 0, w.n_experts) for l in range(L)}
    handle = {}

    def slot_of(l, e):
        return (l * w.n_experts + e + 1) * 65536

    for l in range(L):
        for e in range(w.n_experts):
            handle[slot_of(l, e)] = recs[l][e]
    x = synth.tokens(w).astype(np.float64)

    def layers(absent):
        out = []
        for l in range(L):
            row = np.array([slot_of(l, e) for e in range(w.n_experts)], dtype=np.uint64)
            for (la, e) in absent:
                if la == l:
                    row[e] = 0
            out.append(oracle.LayerInputs(synth.router(w, l), row))
        return out

    full = oracle.moe_stack(x, layers([]), w.top_k, handle.__getitem__, w.hidden, w.inter, grid)
    assert full.miss == [0] * L and full.first_early_out == NO_EARLY_OUT and full.fills == []
    # remove every expert that layer 2 selects, plus one unselected expert of layer 1
    sel2 = sorted(set(full.routes[2].ids.reshape(-1).tolist()))
    unsel1 = sorted(set(range(w.n_experts)) - set(full.routes[1].ids.reshape(-1).tolist()))[0]
    absent = [(2, e) for e in sel2] + [(1, unsel1)]
    part = oracle.moe_stack(x, layers(absent), w.top_k, handle.__getitem__, w.hidden, w.inter, grid,
                            new_slot=slot_of)
    assert part.miss == [0, 0, w.tokens * w.top_k, 0]
    assert part.first_early_out == 2
    assert part.fills == [(2, e) for e in sel2]
    assert np.array_equal(part.x_out, full.x_out)      # the filled chain completes identically
    # brute force: first early-out layer = first layer with a miss
    assert part.first_early_out == min(l for l in range(L) if part.miss[l] > 0)
