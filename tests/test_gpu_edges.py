"""Edge cases of the routed-MoE path on the GPU, each against the oracle:

- an empty prefill chunk (T = 0) with buffers sized for more tokens: nothing runs, the pair
  offsets are all zero, the output and the control block are untouched;
- prefill chunks whose pair counts leave ragged tails in the grouped kernels' token blocks
  and in the router GEMM's token tiles (1, 37 and 300 tokens on the small layer);
- the degenerate routings top-1 (one expert, weight exactly 1) and top-k = number of experts
  (every expert selected), through single-token decode, both prefill paths and the fused
  decode stack.

The shapes are variants of the small layer (hidden 512, 32 experts, top-4, intermediate 128)
so that the oracle finishes in seconds."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from tests._gpu_common import LOGIT_FIXED, REL_TC, REL_F32, OracleSide, check_route, rel_l2, u64  # noqa: E402

TINY = synth.WORKLOADS["tiny"]
DEGENERATE = {
    "top1": replace(TINY, top_k=1),
    "all_experts": replace(TINY, n_experts=16, top_k=16),
}


def _engine():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_moe_expert_rl_gb300 import engine
    return engine


def _prefill(engine, w, m, o, x, path):
    """One prefill chunk on rows x; returns (y, routing checked against the oracle)."""
    T = x.shape[0]
    b = engine.PrefillBuffers.make(m, T)
    y = torch.full_like(x, 7.0)
    engine.enqueue_prefill_route(m, b, 0, x, stacked=False, keep_logits=True)
    engine.enqueue_prefill_experts(m, b, 0, x, y, stacked=False, path=path)
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [0x7FFFFFFF, 0]
    xo = x.double().cpu().numpy()
    r = check_route(b.logits.cpu().numpy(), b.ids.cpu().numpy(), b.weights.cpu().numpy(), u64(b.slots),
                    oracle.router_logits(xo, o.router(0)), o.table_row(0), w.top_k, 0, {})
    offs, ptok, pk = oracle.build_pairs(r.ids, w.n_experts)
    P = T * w.top_k
    assert np.array_equal(b.offs.cpu().numpy().astype(np.uint32), offs)
    assert np.array_equal(b.pair_tok[:P].cpu().numpy().astype(np.uint32), ptok)
    assert np.array_equal(b.pair_k[:P].cpu().numpy(), pk)
    return y.double().cpu().numpy(), o.experts(xo, r.ids, r.weights, r.slots), r


def test_prefill_empty_chunk():
    engine = _engine()
    m = engine.Model(TINY)
    b = engine.PrefillBuffers.make(m, TINY.tokens)
    b.offs.fill_(7)
    x = torch.from_numpy(synth.tokens(TINY)).cuda()
    y = torch.full_like(x, 3.0)
    for path in ("tc", "f32"):
        engine.enqueue_prefill_route(m, b, 0, x[:0], stacked=False)
        engine.enqueue_prefill_experts(m, b, 0, x[:0], y[:0], stacked=False, path=path)
        torch.cuda.synchronize()
        assert int(b.offs.abs().sum()) == 0                     # no pairs: every range empty
        assert bool((y == 3.0).all())
        assert b.ctrl.tolist() == [0x7FFFFFFF, 0] and int(b.miss.sum()) == 0


@pytest.mark.parametrize("T", [1, 37, 300])
@pytest.mark.parametrize("path", ["f32", "tc"])
def test_prefill_ragged_chunks(T, path):
    engine = _engine()
    w = replace(TINY, tokens=T)
    m = engine.Model(w)
    o = OracleSide(m)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    y, y_o, _ = _prefill(engine, w, m, o, x, path)
    assert rel_l2(y, y_o) <= (REL_F32 if path == "f32" else REL_TC)


@pytest.mark.parametrize("name", sorted(DEGENERATE))
def test_degenerate_routing_decode_and_prefill(name):
    engine = _engine()
    w = DEGENERATE[name]
    m = engine.Model(w)
    o = OracleSide(m)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    # single-token decode
    b = engine.DecodeBuffers.make(m)
    y = torch.zeros_like(x)
    for t in range(w.tokens):
        engine.enqueue_decode_token(m, b, x[t], y[t], stacked=False, keep_logits=True)
        torch.cuda.synchronize()
        xo = x[t:t + 1].double().cpu().numpy()
        r = check_route(b.logits[0:1].cpu().numpy(), b.ids[0:1].cpu().numpy(), b.weights[0:1].cpu().numpy(),
                        u64(b.slots[0:1]), oracle.router_logits(xo, o.router(0)), o.table_row(0), w.top_k, 0, {})
        if w.top_k == 1:
            assert float(b.weights[0, 0]) == 1.0
        if w.top_k == w.n_experts:
            assert sorted(r.ids[0].tolist()) == list(range(w.n_experts))
        assert rel_l2(y[t].cpu().numpy(), o.experts(xo, r.ids, r.weights, r.slots)[0]) <= REL_F32
    assert b.ctrl.tolist() == [0x7FFFFFFF, 0]
    # the same tokens as one chunk, on both grouped paths
    for path, tol in (("f32", REL_F32), ("tc", REL_TC)):
        yp, y_o, r = _prefill(engine, w, m, o, x, path)
        assert rel_l2(yp, y_o) <= tol, (path, rel_l2(yp, y_o))


@pytest.mark.parametrize("name", sorted(DEGENERATE))
def test_degenerate_routing_fused_stack(name):
    """Two stacked layers in one moe_decode_stack launch per token, each layer checked against
    the oracle from the GPU's own input to it."""
    engine = _engine()
    w = replace(DEGENERATE[name], n_layers=2)
    m = engine.Model(w)
    o = OracleSide(m)
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    y = torch.zeros_like(x)
    hist = torch.zeros((m.L, w.hidden), dtype=torch.float32, device="cuda")
    for t in range(w.tokens):
        engine.enqueue_decode_token_fused(m, b, x[t], y[t], keep_logits=True, x_hist=hist)
        torch.cuda.synchronize()
        assert b.ctrl.tolist() == [0x7FFFFFFF, 0]
        H = np.concatenate([hist.double().cpu().numpy(), y[t:t + 1].double().cpu().numpy()])
        assert np.array_equal(H[0], x[t].double().cpu().numpy())
        for l in range(m.L):
            xn = oracle.rmsnorm(H[l:l + 1])
            r = check_route(b.logits[l:l + 1].cpu().numpy(), b.ids[l:l + 1].cpu().numpy(),
                            b.weights[l:l + 1].cpu().numpy(), u64(b.slots[l:l + 1]),
                            oracle.router_logits(xn, o.router(l)), o.table_row(l), w.top_k, l, {},
                            logit_tol=LOGIT_FIXED)
            assert rel_l2(H[l + 1] - H[l], o.experts(xn, r.ids, r.weights, r.slots)[0]) <= REL_F32, (t, l)


def test_nan_router_logit_is_flagged():
    """A NaN router logit is refused through RL_DEVERR_NAN in ctrl[1]: it ranks below every
    number, so the selection is the oracle's top-k over the other logits.  In the fused stack
    the NaN partial dot is outside the fixed-point range and raises RL_DEVERR_RANGE instead."""
    engine = _engine()
    from quantized_moe_expert_rl_gb300 import _lib
    w = synth.WORKLOADS["tiny"]
    m = engine.Model(w)
    m.routers[0][3].fill_(float("nan"))
    x = torch.from_numpy(synth.tokens(w)).cuda()
    # decode (rl_route, one token)
    b = engine.DecodeBuffers.make(m)
    y = torch.zeros_like(x)
    engine.enqueue_decode_token(m, b, x[0], y[0], stacked=False, keep_logits=True)
    torch.cuda.synchronize()
    lg = b.logits[0].cpu().numpy()
    assert np.isnan(lg[3]) and int(b.ctrl[1]) & _lib.RL_DEVERR_NAN
    ref = oracle.select_topk(np.where(np.isnan(lg), -np.inf, lg)[None, :], w.top_k)[0]
    assert np.array_equal(b.ids[0].cpu().numpy(), ref) and 3 not in ref.tolist()
    # prefill routing of the chunk
    bp = engine.PrefillBuffers.make(m, w.tokens)
    engine.enqueue_prefill_route(m, bp, 0, x, stacked=False, keep_logits=True)
    torch.cuda.synchronize()
    lgp = bp.logits.cpu().numpy()
    assert int(bp.ctrl[1]) & _lib.RL_DEVERR_NAN
    refp = oracle.select_topk(np.where(np.isnan(lgp), -np.inf, lgp), w.top_k)
    assert np.array_equal(bp.ids.cpu().numpy(), refp)
    # the fused stack
    bf = engine.DecodeBuffers.make(m)
    engine.enqueue_decode_token_fused(m, bf, x[0], y[1])
    torch.cuda.synchronize()
    assert int(bf.ctrl[1]) & _lib.RL_DEVERR_RANGE and not int(bf.ctrl[1]) & _lib.RL_DEVERR_WAIT_TIMEOUT
