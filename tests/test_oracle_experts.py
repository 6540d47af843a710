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


# ----------------------------------------------------------------------------------------------
# The stack recurrence x_{l+1} = x_l + MoE_l(RMSNorm(x_l)), pinned by a closed form.
# Every matrix of every expert is constant (an all-8 codebook row, one scale, one sign for the
# whole matrix) and x starts constant, so x stays a constant vector s_l * 1 and each layer can
# be written out by hand:
#   xn     = s / sqrt(s^2 + eps)                  (RMSNorm of a constant vector)
#   logit_e = r_le * xn   (router rows constant r_le / H), rounded to f32 as the router is
#   top-K by logit; w_k = exp(l_k - l_1) / sum_j exp(l_j - l_1)
#   gate = a_e H xn, up = b_e H xn, h = silu(gate) up, o_e = c_e I h
#   s_{l+1} = s_l + sum_k w_k o_{id_k}
# A dropped residual, a norm taken after the router or not at all, swapped gate/up, a wrong
# selection direction or weights from the wrong logits each change s_{l+1}.
# ----------------------------------------------------------------------------------------------
def _matrix_blocks(n_blocks, d_bits, negative):
    blk = bytes([d_bits & 0xFF, d_bits >> 8]) + bytes([0, 0xFF if negative else 0]) * 32
    return blk * n_blocks


def _fp16_pow2(bits):
    return 2.0 ** (((bits >> 10) & 31) - 15)


def _stack_closed_form(x0, routers, experts, K, H, I, eps):
    """s_l by hand for constant x; routers[l][e] = r_le; experts[l][e] = (a, b, c) values."""
    s = x0
    out = [s]
    sel = []
    for l in range(len(routers)):
        xn = s / math.sqrt(s * s + eps)
        lg = [float(np.float32(r * xn)) for r in routers[l]]
        order = sorted(range(len(lg)), key=lambda e: (-lg[e], e))[:K]
        ex = [math.exp(lg[e] - lg[order[0]]) for e in order]
        tot = 0.0
        for v in ex:
            tot += v
        y = 0.0
        for j, e in enumerate(order):
            a, b, c = experts[l][e]
            g, u = a * H * xn, b * H * xn
            h = g / (1 + math.exp(-g)) * u
            y += (ex[j] / tot) * (c * I * h)
        s = s + y
        out.append(s)
        sel.append(order)
    return out, sel


def _stack_case(x0, routers, specs, K, H=256, I=256, eps=1e-6):
    grid = np.full((256, 8), 8, dtype=np.int8)
    L, E = len(routers), len(routers[0])
    nb = H * I // 256
    recs, vals, layers = {}, [], []
    for l in range(L):
        row = np.zeros(E, dtype=np.uint64)
        vl = []
        for e in range(E):
            mats = specs[l][e]           # ((d_bits, negative) for gate, up, down)
            recs[(l * E + e + 1) * 4096] = np.frombuffer(b"".join(_matrix_blocks(nb, *m) for m in mats),
                                                         dtype=np.uint8)
            row[e] = (l * E + e + 1) * 4096
            vl.append(tuple(8 * _fp16_pow2(db) * (-1.0 if neg else 1.0) for db, neg in mats))
        vals.append(vl)
        wr = np.repeat(np.asarray(routers[l], dtype=np.float32)[:, None] / np.float32(H), H, axis=1)
        layers.append(oracle.LayerInputs(wr, row))
    x = np.full((1, H), x0)
    res = oracle.moe_stack(x, layers, K, recs.__getitem__, H, I, grid, eps=eps)
    expect, sel = _stack_closed_form(x0, routers, vals, K, H, I, eps)
    return res, expect, sel


def test_stack_recurrence_closed_form():
    # fp16 scales: 0x2000 = 2^-7, 0x1C00 = 2^-8, 0x1800 = 2^-9, 0x1400 = 2^-10, 0x0C00 = 2^-12
    routers = [[0.75, 0.5, -0.25, -0.5],      # x > 0: layer 0 picks experts 0, 1
               [-0.5, 0.25, 0.5, 1.0],        # layer 1 picks 3, 2 while x > 0
               [0.125, -1.0, 0.5, -0.75]]     # the sign of x decides layer 2
    specs = [
        [((0x1C00, False), (0x1800, False), (0x0C00, True)), ((0x1800, False), (0x1C00, True), (0x0C00, False)),
         ((0x1400, False), (0x1400, False), (0x0C00, False)), ((0x1400, True), (0x1400, False), (0x0C00, False))],
        [((0x1800, False), (0x1800, False), (0x0C00, False)), ((0x1400, False), (0x1800, False), (0x0C00, True)),
         ((0x1C00, True), (0x1800, False), (0x0C00, False)), ((0x1800, False), (0x1C00, False), (0x0C00, True))],
        [((0x1800, False), (0x1400, False), (0x0C00, False)), ((0x1C00, False), (0x1800, True), (0x0C00, True)),
         ((0x1400, False), (0x1C00, False), (0x0C00, True)), ((0x1800, True), (0x1800, False), (0x0C00, False))],
    ]
    for x0 in (0.75, -2.0):
        res, expect, sel = _stack_case(x0, routers, specs, K=2)
        assert [r.ids[0].tolist() for r in res.routes] == sel
        for l, xi in enumerate(res.x_in):
            assert np.allclose(xi, expect[l], rtol=1e-12, atol=0), (x0, l)
        assert np.allclose(res.x_out, expect[-1], rtol=1e-12, atol=0)
        # the state moves by more than the tolerance every layer, and not by the MoE term alone
        for l in range(3):
            assert abs(expect[l + 1] - expect[l]) > 1e-6 * abs(expect[l + 1])
            assert abs(expect[l + 1] - (expect[l + 1] - expect[l])) > 1e-3
    # the two starting signs route layer 0 differently, and some later layer selects other experts
    r_pos = _stack_case(0.75, routers, specs, K=2)[2]
    r_neg = _stack_case(-2.0, routers, specs, K=2)[2]
    assert r_pos[0] != r_neg[0]
    assert len({tuple(s) for s in r_pos}) >= 2 and len({tuple(s) for s in r_neg}) >= 2


def test_stack_closed_form_rejects_planted_mistakes():
    """The hand-written recurrence above is sensitive to each plausible oracle mistake: the
    values a mistaken recurrence would give differ from the closed form."""
    H, I, eps = 256, 256, 1e-6
    routers = [[0.75, 0.5, -0.25, -0.5], [-0.5, 0.25, 0.5, 1.0]]
    vals = [[(2 ** -5, 2 ** -6, -(2 ** -9)), (2 ** -6, -(2 ** -5), 2 ** -9), (2 ** -7, 2 ** -7, 2 ** -9),
             (-(2 ** -7), 2 ** -7, 2 ** -9)]] * 2
    good, _ = _stack_closed_form(0.75, routers, vals, 2, H, I, eps)

    def variant(residual=True, norm=True, swap=False):
        s = 0.75
        for l in range(2):
            xn = s / math.sqrt(s * s + eps) if norm else s
            lg = [float(np.float32(r * xn)) for r in routers[l]]
            order = sorted(range(4), key=lambda e: (-lg[e], e))[:2]
            ex = [math.exp(lg[e] - lg[order[0]]) for e in order]
            y = 0.0
            for j, e in enumerate(order):
                a, b, c = vals[l][e]
                if swap:
                    a, b = b, a
                g, u = a * H * xn, b * H * xn
                y += ex[j] / sum(ex) * (c * I * g / (1 + math.exp(-g)) * u)
            s = s + y if residual else y
        return s

    assert math.isclose(variant(), good[-1], rel_tol=1e-13)
    for bad in (variant(residual=False), variant(norm=False), variant(swap=True)):
        assert not math.isclose(bad, good[-1], rel_tol=1e-6)
