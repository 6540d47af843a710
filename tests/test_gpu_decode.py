"""Decode parity on the GPU: single-layer decode (sampled tokens of the 1000), the 48-layer
stack through the same per-token CUDA graphs bench.py times (checked layer by layer against
the oracle from the GPU's own layer inputs), the tie rule on exactly equal logits, slot-order
invariance and the early-out path."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from tests._gpu_common import LOGIT_FIXED, REL_F32, OracleSide, check_route, rel_l2, u64  # noqa: E402


def _engine():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_moe_expert_rl_gb300 import engine
    return engine


@pytest.fixture(scope="module")
def layer_model():
    engine = _engine()
    w = synth.WORKLOADS["decode_layer"]
    m = engine.Model(w)
    return w, m, OracleSide(m)


def test_decode_layer_sampled_tokens(layer_model):
    """200 of the 1000 single-layer decode tokens, each run on its own through rl_route +
    moe_decode: routing bit-exact on the GPU's logits (logits within LOGIT_ROUTE), outputs
    within the f32 bound, no near tie at this seed."""
    engine = _engine()
    w, m, o = layer_model
    b = engine.DecodeBuffers.make(m)
    sample = np.unique(np.concatenate([np.arange(0, w.tokens, 5), [w.tokens - 1]]))
    x = torch.from_numpy(synth.tokens(w, 0, w.tokens)).cuda()
    y = torch.zeros_like(x)
    n = len(sample)
    lg = torch.zeros((n, w.n_experts), device="cuda")
    ids = torch.zeros((n, w.top_k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((n, w.top_k), device="cuda")
    sl = torch.zeros((n, w.top_k), dtype=torch.int64, device="cuda")
    for i, t in enumerate(sample):
        engine.enqueue_decode_token(m, b, x[t], y[t], stacked=False, keep_logits=True)
        lg[i].copy_(b.logits[0])
        ids[i].copy_(b.ids[0])
        wts[i].copy_(b.weights[0])
        sl[i].copy_(b.slots[0])
    torch.cuda.synchronize()
    assert int(b.miss[0]) == 0 and b.ctrl.tolist() == [0x7FFFFFFF, 0]
    xo = x[torch.from_numpy(sample).cuda()].double().cpu().numpy()
    rep = {}
    r = check_route(lg.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy(), u64(sl),
                    oracle.router_logits(xo, o.router(0)), o.table_row(0), w.top_k, 0, rep)
    y_o = o.experts(xo, r.ids, r.weights, r.slots)
    yg = y[torch.from_numpy(sample).cuda()].double().cpu().numpy()
    errs = [rel_l2(yg[i], y_o[i]) for i in range(n)]
    print(f"decode_layer: {n} tokens, worst rel L2 {max(errs):.2e}, logit err {rep['logit_err']:.2e}, "
          f"near ties {rep.get('near_ties', 0)}")
    assert max(errs) <= REL_F32
    assert rep.get("near_ties", 0) == 0


def test_decode_layer_fused(layer_model):
    """moe_decode_layer (router and experts of one token in one launch, no norm, no residual)
    on 200 of the 1000 single-layer tokens: routing bit-exact on the GPU's own logits, logits
    within the fused kernel's bound of the row scale (fixed-point sums across CTAs), outputs
    within the f32 bound of the oracle, and the ids of rl_route + moe_decode except at a
    genuine near tie."""
    engine = _engine()
    w, m, o = layer_model
    b, bc = engine.DecodeBuffers.make(m), engine.DecodeBuffers.make(m)
    sample = np.unique(np.concatenate([np.arange(3, w.tokens, 5), [w.tokens - 1]]))
    x = torch.from_numpy(synth.tokens(w, 0, w.tokens)).cuda()
    n = len(sample)
    y = torch.zeros((n, w.hidden), device="cuda")
    yc = torch.zeros((n, w.hidden), device="cuda")
    lg = torch.zeros((n, w.n_experts), device="cuda")
    ids = torch.zeros((n, w.top_k), dtype=torch.int32, device="cuda")
    idc = torch.zeros((n, w.top_k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((n, w.top_k), device="cuda")
    sl = torch.zeros((n, w.top_k), dtype=torch.int64, device="cuda")
    for i, t in enumerate(sample):
        engine.enqueue_decode_layer_fused(m, b, x[t], y[i], keep_logits=True)
        lg[i].copy_(b.logits[0])
        ids[i].copy_(b.ids[0])
        wts[i].copy_(b.weights[0])
        sl[i].copy_(b.slots[0])
        engine.enqueue_decode_token(m, bc, x[t], yc[i], stacked=False)
        idc[i].copy_(bc.ids[0])
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [0x7FFFFFFF, 0] and int(b.miss[0]) == 0
    xo = x[torch.from_numpy(sample).cuda()].double().cpu().numpy()
    rep = {}
    r = check_route(lg.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy(), u64(sl),
                    oracle.router_logits(xo, o.router(0)), o.table_row(0), w.top_k, 0, rep, logit_tol=LOGIT_FIXED)
    y_o = o.experts(xo, r.ids, r.weights, r.slots)
    yg = y.double().cpu().numpy()
    errs = [rel_l2(yg[i], y_o[i]) for i in range(n)]
    same = np.all(ids.cpu().numpy() == idc.cpu().numpy(), axis=1)
    yd = yc.double().cpu().numpy()
    for i in np.nonzero(same)[0]:
        assert rel_l2(yg[i], yd[i]) <= REL_F32, i
    print(f"decode_layer fused: {n} tokens, worst rel L2 {max(errs):.2e}, logit err {rep['logit_err']:.2e}, "
          f"near ties {rep.get('near_ties', 0)}, ids as rl_route on {int(same.sum())}/{n}")
    assert max(errs) <= REL_F32
    assert rep.get("near_ties", 0) <= 1 and int(same.sum()) >= n - 1


def test_decode_graph_equals_eager(layer_model):
    engine = _engine()
    w, m, _ = layer_model
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w, 0, 8)).cuda()
    y_e, y_g = torch.zeros_like(x), torch.zeros_like(x)
    for t in range(8):
        engine.enqueue_decode_token(m, b, x[t], y_e[t], stacked=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gs = []
    for t in range(8):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            engine.enqueue_decode_token(m, b, x[t], y_g[t], stacked=False)
        gs.append(g)
    for g in gs:
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_e, y_g)


@pytest.fixture(scope="module")
def stack_model():
    engine = _engine()
    w = synth.WORKLOADS["decode_stack"]
    m = engine.Model(w)
    return w, m, OracleSide(m)


def test_decode_stack_layer_by_layer(stack_model):
    """Three tokens through all 48 layers with the per-token graphs; every layer is checked
    against the oracle computed from the GPU's own input to that layer (ids and slots
    bit-exact on the GPU's logits, layer output within the f32 bound)."""
    engine = _engine()
    w, m, o = stack_model
    b = engine.DecodeBuffers.make(m)
    toks = [0, 128, w.tokens - 1]
    x = torch.from_numpy(synth.tokens(w, 0, w.tokens)).cuda()
    y = torch.zeros_like(x)
    hist = torch.zeros((len(toks), m.L + 1, w.hidden), dtype=torch.float32, device="cuda")
    logits = torch.zeros((len(toks), m.L, w.n_experts), dtype=torch.float32, device="cuda")
    ids = torch.zeros((len(toks), m.L, w.top_k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((len(toks), m.L, w.top_k), dtype=torch.float32, device="cuda")
    slots = torch.zeros((len(toks), m.L, w.top_k), dtype=torch.int64, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for i, t in enumerate(toks):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            engine.enqueue_decode_token(m, b, x[t], y[t], stacked=True, keep_logits=True, x_hist=hist[i])
        g.replay()
        torch.cuda.synchronize()
        hist[i, m.L].copy_(y[t])
        logits[i].copy_(b.logits)
        ids[i].copy_(b.ids)
        wts[i].copy_(b.weights)
        slots[i].copy_(b.slots)
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [0x7FFFFFFF, 0] and int(b.miss.sum()) == 0
    H = hist.double().cpu().numpy()
    rep, worst = {}, 0.0
    for i, t in enumerate(toks):
        assert np.array_equal(H[i, 0], synth.tokens(w, t, 1)[0].astype(np.float64))
        for l in range(m.L):
            xl = H[i, l:l + 1]
            xn = oracle.rmsnorm(xl)
            r = check_route(logits[i, l:l + 1].cpu().numpy(), ids[i, l:l + 1].cpu().numpy(),
                            wts[i, l:l + 1].cpu().numpy(), u64(slots[i, l:l + 1]),
                            oracle.router_logits(xn, o.router(l)), o.table_row(l), w.top_k, l, rep)
            y_o = o.experts(xn, r.ids, r.weights, r.slots)
            err = rel_l2(H[i, l + 1] - H[i, l], y_o[0])
            worst = max(worst, err)
            assert err <= REL_F32, (t, l, err)
    print(f"stack: worst per-layer rel L2 {worst:.2e}, logit err {rep['logit_err']:.2e}, "
          f"near ties {rep.get('near_ties', 0)}")
    assert rep.get("near_ties", 0) == 0


def test_tie_rule_on_equal_logits():
    """Duplicated router rows give bit-equal logits on the GPU (same reduction for every
    row): the lower expert index must come first, as in the oracle."""
    engine = _engine()
    w = synth.WORKLOADS["tiny"]
    m = engine.Model(w)
    wr = m.routers[0].clone()
    # make experts 5, 9, 20 copies of expert 2's row and 30 a copy of 11's
    for dst, src in ((5, 2), (9, 2), (20, 2), (30, 11)):
        m.routers[0][dst].copy_(m.routers[0][src])
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    y = torch.zeros_like(x)
    seen_tie = False
    for t in range(w.tokens):
        engine.enqueue_decode_token(m, b, x[t], y[t], stacked=False, keep_logits=True)
        torch.cuda.synchronize()
        lg = b.logits[0].cpu().numpy()
        assert lg[5] == lg[2] and lg[9] == lg[2] and lg[20] == lg[2] and lg[30] == lg[11]
        ref = oracle.select_topk(lg[None, :], w.top_k)[0]
        assert np.array_equal(b.ids[0].cpu().numpy(), ref)
        seen_tie |= len(set(ref.tolist()) & {2, 5, 9, 20}) > 1
    m.routers[0].copy_(wr)
    # the top logit of some token must sit in a tie group; force it if the data did not
    if not seen_tie:
        for dst in (5, 9, 20):
            m.routers[0][dst].copy_(m.routers[0][int(b.ids[0, 0])])
        engine.enqueue_decode_token(m, b, x[w.tokens - 1], y[0], stacked=False, keep_logits=True)
        torch.cuda.synchronize()
        ref = oracle.select_topk(b.logits[0].cpu().numpy()[None, :], w.top_k)[0]
        assert np.array_equal(b.ids[0].cpu().numpy(), ref)


def test_slot_order_invariance():
    engine = _engine()
    w = synth.WORKLOADS["tiny"]
    outs = []
    for perm in (False, True):
        m = engine.Model(w, slot_perm=perm)
        b = engine.DecodeBuffers.make(m)
        x = torch.from_numpy(synth.tokens(w)).cuda()
        y = torch.zeros_like(x)
        ids, ws_, sl = [], [], []
        for t in range(w.tokens):
            engine.enqueue_decode_token(m, b, x[t], y[t], stacked=False)
            torch.cuda.synchronize()
            ids.append(b.ids[0].cpu().numpy().copy())
            ws_.append(b.weights[0].cpu().numpy().copy())
            sl.append([m.expert_of_addr()[int(v)] for v in u64(b.slots[0])])
        outs.append((np.array(ids), np.array(ws_), y.cpu().numpy(), sl))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][2], outs[1][2])           # bit-identical outputs
    assert outs[0][3] == outs[1][3]                          # slots name the same experts


def test_decode_early_out():
    """A layer that selects an absent expert raises the flag; the experts of that layer and
    every later layer are skipped; the miss count is exact."""
    engine = _engine()
    w = replace(synth.WORKLOADS["tiny"], n_layers=3)
    m = engine.Model(w)
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w, 0, 1)).cuda()
    y = torch.zeros_like(x)
    engine.enqueue_decode_token(m, b, x[0], y[0], stacked=True)
    torch.cuda.synchronize()
    ids1 = b.ids[1].cpu().numpy().copy()
    # remove two of layer 1's selected experts
    for e in ids1[:2]:
        m.table_host[1, e] = 0
    m.table[1].copy_(torch.from_numpy(m.table_host[1].view(np.int64).copy()))
    b.miss.zero_()
    b.ctrl.copy_(torch.tensor([0x7FFFFFFF, 0], dtype=torch.int32))
    engine.enqueue_decode_token(m, b, x[0], y[0], stacked=True, x_hist=(hist := torch.zeros(3, w.hidden).cuda()))
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [1, 0]
    assert b.miss.tolist() == [0, 2, 0]
    # layer 0 ran, layer 1's experts and layer 2 were skipped: the output is layer 1's input
    assert torch.equal(y[0], hist[1])


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def test_decode_stack_fused_vs_chain(stack_model):
    """moe_decode_stack (one launch per token for all 48 layers) against the per-layer chain
    rl_route + moe_decode.  The fused launch sums every router row across its CTAs in 64-bit
    fixed point, so its logits differ from rl_route's f32 dots in the last bits only: at the
    first layer (same input) within 1e-6 of the row scale; the selections equal except at a
    genuine near tie (where the two paths part); the token outputs within the f32 bound.  Every
    fused layer of the first token, and every 4th of the others, matches the oracle from its
    own input.  The pre-gated prefetch changes no result: with and without it the fused runs
    are bit-identical, and its hit counts follow from the GPU's own layer inputs."""
    engine = _engine()
    w, m, o = stack_model
    toks = [0, 77, w.tokens - 1]
    x = torch.from_numpy(synth.tokens(w, 0, w.tokens)).cuda()
    outs = {}
    hits = torch.zeros((len(toks), m.L), dtype=torch.int32, device="cuda")
    for mode in ("chain", "fused", "fused_pregate"):
        b = engine.DecodeBuffers.make(m)
        hist = torch.zeros((len(toks), m.L, w.hidden), device="cuda")
        res = []
        for i, t in enumerate(toks):
            y = torch.zeros(w.hidden, device="cuda")
            if mode == "chain":
                engine.enqueue_decode_token(m, b, x[t], y, stacked=True, keep_logits=True, x_hist=hist[i])
            else:
                pg = 32 if mode == "fused_pregate" else 0
                engine.enqueue_decode_token_fused(m, b, x[t], y, keep_logits=True, x_hist=hist[i], pregate=pg,
                                                  pregate_hits=hits[i] if pg else None)
            torch.cuda.synchronize()
            res.append([_bits(v) for v in (b.logits, b.ids, b.weights, b.slots, y)])
        assert b.ctrl.tolist() == [0x7FFFFFFF, 0] and int(b.miss.sum()) == 0
        outs[mode] = (res, _bits(hist), hist.double().cpu().numpy())
    # the prefetch never changes a result
    for ra, rb in zip(outs["fused"][0], outs["fused_pregate"][0]):
        for name, a_, b_ in zip(("logits", "ids", "weights", "slots", "y"), ra, rb):
            assert torch.equal(a_, b_), name
    assert torch.equal(outs["fused"][1], outs["fused_pregate"][1])
    # fused against chain
    for i in range(len(toks)):
        rc, rf = outs["chain"][0][i], outs["fused"][0][i]
        lc, lf = rc[0].view(torch.float32).double().numpy(), rf[0].view(torch.float32).double().numpy()
        assert np.max(np.abs(lc[0] - lf[0])) <= 1e-6 * np.max(np.abs(lc[0])), i
        ic, if_ = rc[1].numpy(), rf[1].numpy()
        diff = np.nonzero(np.any(ic != if_, axis=1))[0]
        if len(diff):   # only a genuine near tie may differ; the paths part there
            l = int(diff[0])
            for a_, b_ in zip(ic[l], if_[l]):
                if a_ != b_:
                    assert abs(lc[l][a_] - lc[l][b_]) <= 1e-5 * np.max(np.abs(lc[l])), (i, l)
            print(f"token {toks[i]}: near tie at layer {l}")
            continue
        assert torch.equal(rc[3], rf[3]), i
        yc, yf = rc[4].view(torch.float32).double().numpy(), rf[4].view(torch.float32).double().numpy()
        assert rel_l2(yf, yc) <= REL_F32, (i, rel_l2(yf, yc))
    # pre-gate hits: layer l's experts found in the top-32 of router l applied at layer l-1,
    # recomputed on the host from the GPU's own layer inputs (f32 logits; near ties may move one)
    Hh = outs["fused_pregate"][2]
    hits = hits.cpu().numpy()
    for i in range(len(toks)):
        ids = outs["fused_pregate"][0][i][1].numpy()
        for l in range(1, m.L):
            xn = oracle.rmsnorm(Hh[i][l - 1:l])
            lg = oracle.router_logits(xn, o.router(l))[0]
            pred = set(np.lexsort((np.arange(len(lg)), -lg))[:32].tolist())
            want = len(set(ids[l].tolist()) & pred)
            assert abs(int(hits[i, l]) - want) <= 1, (i, l, int(hits[i, l]), want)
    rate = hits[:, 1:].mean() / w.top_k
    print(f"pre-gate (top-32) hit rate {rate:.2f}")
    assert rate > 0.5
    # the fused layers against the oracle, each from its own layer input
    rep = {}
    for i in range(len(toks)):
        H = outs["fused"][2][i]
        y_last = outs["fused"][0][i][4].view(torch.float32).double().numpy()
        r_all = outs["fused"][0][i]
        for l in range(0, m.L, 1 if i == 0 else 4):
            xn = oracle.rmsnorm(H[l:l + 1])
            lg = r_all[0].view(torch.float32).numpy()[l:l + 1]
            ids = r_all[1].numpy()[l:l + 1]
            wts = r_all[2].view(torch.float32).numpy()[l:l + 1]
            sl = r_all[3].numpy().view(np.uint64)[l:l + 1]
            r = check_route(lg, ids, wts, sl, oracle.router_logits(xn, o.router(l)), o.table_row(l), w.top_k, l, rep,
                            logit_tol=LOGIT_FIXED)
            y_o = o.experts(xn, r.ids, r.weights, r.slots)
            x_next = H[l + 1] if l + 1 < m.L else y_last
            assert rel_l2(x_next - H[l], y_o[0]) <= REL_F32, (i, l)
    print(f"fused stack: logit err {rep['logit_err']:.2e}, near ties {rep.get('near_ties', 0)}")
    assert rep.get("near_ties", 0) <= 1


def test_decode_stack_bounded_residency():
    """Bounded residency through the fused stack: each token stops at the first layer that
    selects an absent expert, with the exact miss count; the host fills that layer's missing
    experts and resumes.  Outputs and selections equal those of a fully resident model bit
    for bit, and the early-out layers follow from the selections and the residency."""
    engine = _engine()
    base = replace(synth.WORKLOADS["tiny"], n_layers=6)
    wb = replace(base, n_resident=26)
    m_full, m_b = engine.Model(base), engine.Model(wb)
    b_full, b_b = engine.DecodeBuffers.make(m_full), engine.DecodeBuffers.make(m_b)
    x = torch.from_numpy(synth.tokens(base, 0, base.tokens)).cuda()
    resident = np.stack([synth.resident_mask(wb, l).astype(bool) for l in range(wb.n_layers)])
    n_early = 0
    for t in range(base.tokens):
        y_full = torch.zeros(base.hidden, device="cuda")
        y_b = torch.zeros(base.hidden, device="cuda")
        engine.enqueue_decode_token_fused(m_full, b_full, x[t], y_full)
        b_b.miss.zero_()
        st = engine.run_bounded_decode_token(m_b, b_b, x[t], y_b)
        torch.cuda.synchronize()
        assert torch.equal(_bits(y_full), _bits(y_b)), t
        assert torch.equal(_bits(b_full.ids), _bits(b_b.ids)) and torch.equal(_bits(b_full.weights), _bits(b_b.weights))
        ids = b_full.ids.cpu().numpy()
        exp_miss, exp_early, exp_fill = [], [], []
        for l in range(wb.n_layers):
            miss = [int(e) for e in ids[l] if not resident[l, e]]
            exp_miss.append(len(miss))
            if miss:
                exp_early.append(l)
                exp_fill += [(l, e) for e in sorted(set(miss))]
                resident[l, list(set(miss))] = True
        assert b_b.miss.tolist() == exp_miss, t
        assert st.early_outs == exp_early and st.filled == exp_fill, t
        assert b_b.ctrl.tolist() == [0x7FFFFFFF, 0]
        n_early += len(st.early_outs)
    print(f"bounded fused decode: {n_early} early-outs over {base.tokens} tokens")
    assert n_early > 0


def test_decode_stack_range_flag():
    """A residual stream far outside the fixed-point range of the fused kernel's router sums
    (|partial dot| >= 2^19) raises RL_DEVERR_RANGE in ctrl[1] and the launch still completes;
    an input of ordinary scale leaves ctrl[1] at 0."""
    engine = _engine()
    from quantized_moe_expert_rl_gb300 import _lib
    w = replace(synth.WORKLOADS["tiny"], n_layers=3)
    m = engine.Model(w)
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w, 0, 1)).cuda()[0]
    y = torch.zeros(w.hidden, device="cuda")
    engine.enqueue_decode_token_fused(m, b, x, y)
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [0x7FFFFFFF, 0]
    b.ctrl.copy_(torch.tensor([0x7FFFFFFF, 0], dtype=torch.int32))
    engine.enqueue_decode_token_fused(m, b, x * 1e9, y)
    torch.cuda.synchronize()
    c = b.ctrl.tolist()
    assert c[1] & _lib.RL_DEVERR_RANGE and not (c[1] & _lib.RL_DEVERR_WAIT_TIMEOUT), c


def test_decode_stack_bounded_lookahead():
    """Bounded residency with lookahead fills: at each stop the next layer is routed on its
    input and the layer after it pre-gated from the same input, and their absent experts are
    filled before the stack restarts.  The outputs stay bit-identical to a fully resident run;
    the stack stops no more often than without lookahead, and every expert any layer selected
    ends up resident."""
    engine = _engine()
    base = replace(synth.WORKLOADS["tiny"], n_layers=6)
    wb = replace(base, n_resident=26)
    m_full = engine.Model(base)
    b_full = engine.DecodeBuffers.make(m_full)
    x = torch.from_numpy(synth.tokens(base, 0, base.tokens)).cuda()
    stops = {}
    for look in (False, True):
        m_b = engine.Model(wb)
        b_b = engine.DecodeBuffers.make(m_b)
        n_stop = n_pre = 0
        for t in range(base.tokens):
            y_full = torch.zeros(base.hidden, device="cuda")
            y_b = torch.zeros(base.hidden, device="cuda")
            engine.enqueue_decode_token_fused(m_full, b_full, x[t], y_full)
            b_b.miss.zero_()
            st = engine.run_bounded_decode_token(m_b, b_b, x[t], y_b, lookahead=look)
            torch.cuda.synchronize()
            assert torch.equal(_bits(y_full), _bits(y_b)), (look, t)
            assert torch.equal(_bits(b_full.ids), _bits(b_b.ids)), (look, t)
            ids = b_full.ids.cpu().numpy()
            for l in range(wb.n_layers):
                assert all(m_b.resident[l, int(e)] for e in ids[l]), (look, t, l)
            n_stop += len(st.early_outs)
            n_pre += len(st.prefetched)
            if not look:
                assert st.prefetched == []
        stops[look] = (n_stop, n_pre)
    print(f"bounded decode stops without / with lookahead: {stops[False][0]} / {stops[True][0]}, "
          f"{stops[True][1]} experts filled ahead")
    assert stops[True][0] <= stops[False][0] and stops[True][1] > 0


def test_decode_stack_device_fill():
    """Bounded residency with the fills done inside the fused launch (moe_decode_stack_fill):
    no stop, the same per-layer miss counts and fills as the stop / fill / resume flow, outputs
    bit-identical to a fully resident model."""
    engine = _engine()
    base = replace(synth.WORKLOADS["tiny"], n_layers=6)
    wb = replace(base, n_resident=26)
    m_full, m_h, m_d = engine.Model(base), engine.Model(wb), engine.Model(wb)
    b_full, b_h, b_d = (engine.DecodeBuffers.make(m) for m in (m_full, m_h, m_d))
    x = torch.from_numpy(synth.tokens(base, 0, base.tokens)).cuda()
    filled = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_host_fills = 0
    for t in range(base.tokens):
        y_full, y_h, y_d = (torch.zeros(base.hidden, device="cuda") for _ in range(3))
        engine.enqueue_decode_token_fused(m_full, b_full, x[t], y_full)
        b_h.miss.zero_()
        st = engine.run_bounded_decode_token(m_h, b_h, x[t], y_h)
        b_d.miss.zero_()
        engine.run_bounded_decode_token_device(m_d, b_d, x[t], y_d, filled)
        torch.cuda.synchronize()
        assert b_d.ctrl.tolist() == [0x7FFFFFFF, 0], t
        assert torch.equal(_bits(y_full), _bits(y_d)), t
        assert torch.equal(_bits(y_h), _bits(y_d)), t
        assert b_h.miss.tolist() == b_d.miss.tolist(), t
        assert torch.equal(_bits(b_h.ids), _bits(b_d.ids)), t
        # the two models have their own pools: compare slots as offsets into them
        oh = b_h.slots.cpu() - m_h.pool.data_ptr()
        od = b_d.slots.cpu() - m_d.pool.data_ptr()
        assert torch.equal(oh, od), t
        n_host_fills += len(st.filled)
    m_d.sync_residency_from_device()
    assert np.array_equal(m_d.resident, m_h.resident)
    assert int(filled.item()) == n_host_fills > 0
    print(f"device fills inside the fused launch: {n_host_fills} experts over {base.tokens} tokens, no stop")


def test_decode_stack_bounded_full_shape(stack_model):
    """Bounded residency at the full decode-stack shape: 48 layers x 512 experts with 435 of
    them resident per layer (seeded), three tokens in turn from that residency, through the
    stop / fill / resume flow and through the fills done inside the fused launch.  Both give
    the bits of the fully resident model; the per-layer miss counts, the stopping layers and
    the filled experts follow exactly from the fully resident run's selections and the
    residency so far; sampled layers of the first token match the oracle from their own
    inputs."""
    engine = _engine()
    w, m_full, _ = stack_model
    wb = replace(w, n_resident=435)
    m_b = engine.Model(wb)
    ob = OracleSide(m_b)    # the bounded model's slot addresses point into its own pool
    b_full, b_b = engine.DecodeBuffers.make(m_full), engine.DecodeBuffers.make(m_b)
    toks = [0, 1, 2]
    x = torch.from_numpy(synth.tokens(w, 0, 3)).cuda()
    seeded = np.stack([synth.resident_mask(wb, l).astype(bool) for l in range(wb.n_layers)])
    summary = {}
    for mode in ("host", "device"):
        m_b.reset_residency()
        resident = seeded.copy()
        filled = torch.zeros(1, dtype=torch.int32, device="cuda")
        n_stop = n_fill = 0
        for i, t in enumerate(toks):
            y_full = torch.zeros(w.hidden, device="cuda")
            y_b = torch.zeros(w.hidden, device="cuda")
            hist = torch.zeros((m_b.L, w.hidden), device="cuda")
            engine.enqueue_decode_token_fused(m_full, b_full, x[i], y_full)
            b_b.miss.zero_()
            if mode == "host":
                st = engine.run_bounded_decode_token(m_b, b_b, x[i], y_b, x_hist=hist)
            else:
                engine.run_bounded_decode_token_device(m_b, b_b, x[i], y_b, filled, x_hist=hist)
            torch.cuda.synchronize()
            assert b_b.ctrl.tolist() == [0x7FFFFFFF, 0], (mode, t)
            assert torch.equal(_bits(y_full), _bits(y_b)), (mode, t)
            assert torch.equal(_bits(b_full.ids), _bits(b_b.ids)), (mode, t)
            assert torch.equal(_bits(b_full.weights), _bits(b_b.weights)), (mode, t)
            ids = b_full.ids.cpu().numpy()
            exp_miss, exp_stop, exp_fill = [], [], []
            for l in range(wb.n_layers):
                miss = [int(e) for e in ids[l] if not resident[l, e]]
                exp_miss.append(len(miss))
                if miss:
                    exp_stop.append(l)
                    exp_fill += [(l, e) for e in sorted(set(miss))]
                    resident[l, sorted(set(miss))] = True
            assert b_b.miss.tolist() == exp_miss, (mode, t)
            if mode == "host":
                assert st.early_outs == exp_stop and st.filled == exp_fill, (mode, t)
                n_stop += len(st.early_outs)
            n_fill += len(exp_fill)
            if i == 0:
                # sampled layers of the first token against the oracle from their own inputs
                H = hist.double().cpu().numpy()
                y_last = y_b.double().cpu().numpy()
                sl = u64(b_b.slots)
                wts = b_b.weights.cpu().numpy()
                for l in (0, 17, wb.n_layers - 1):
                    xn = oracle.rmsnorm(H[l:l + 1])
                    y_o = oracle.moe_experts(xn, ids[l:l + 1], wts[l:l + 1].astype(np.float64), sl[l:l + 1],
                                             ob.record, w.hidden, w.inter, ob.grid)
                    x_next = H[l + 1] if l + 1 < wb.n_layers else y_last
                    assert rel_l2(x_next - H[l], y_o[0]) <= REL_F32, (mode, l)
        if mode == "device":
            assert int(filled.item()) == n_fill
            m_b.sync_residency_from_device()
        assert np.array_equal(m_b.resident, resident), mode
        summary[mode] = (n_stop, n_fill)
    print(f"bounded full-shape decode: {summary['host'][0]} stops and {summary['host'][1]} fills over "
          f"{len(toks)} tokens; device fills {summary['device'][1]}, no stop")
    assert summary["host"][1] == summary["device"][1] > 0
