"""Parity of every entry point on the tiny workload (H=512, E=32, K=4, I=128, 4 tokens) against
the oracle: as 4 single-token decode calls and as one 4-token prefill chunk."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from tests._gpu_common import REL_TC, REL_F32, OracleSide, check_route, rel_l2, u64  # noqa: E402


@pytest.fixture(scope="module")
def tiny():
    from quantized_moe_expert_rl_gb300 import engine
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    w = synth.WORKLOADS["tiny"]
    model = engine.Model(w)
    return w, model, OracleSide(model)


def test_decode_tokens(tiny):
    from quantized_moe_expert_rl_gb300 import engine
    w, model, o = tiny
    b = engine.DecodeBuffers.make(model)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    y = torch.zeros_like(x)
    rep = {}
    for t in range(w.tokens):
        engine.enqueue_decode_token(model, b, x[t], y[t], stacked=False, keep_logits=True)
        torch.cuda.synchronize()
        xo = x[t:t + 1].double().cpu().numpy()
        lg64 = oracle.router_logits(xo, o.router(0))
        r = check_route(b.logits[0:1].cpu().numpy(), b.ids[0:1].cpu().numpy(), b.weights[0:1].cpu().numpy(),
                        u64(b.slots[0:1]), lg64, o.table_row(0), w.top_k, 0, rep)
        y_o = o.experts(xo, r.ids, r.weights, r.slots)
        assert rel_l2(y[t].cpu().numpy(), y_o[0]) <= REL_F32
    assert rep["near_ties"] == 0
    assert int(b.miss[0]) == 0 and int(b.ctrl[0]) == 0x7FFFFFFF and int(b.ctrl[1]) == 0


@pytest.mark.parametrize("path", ["f32", "tc"])
def test_prefill_chunk(tiny, path):
    from quantized_moe_expert_rl_gb300 import engine
    w, model, o = tiny
    T = w.tokens
    b = engine.PrefillBuffers.make(model, T)
    x = torch.from_numpy(synth.tokens(w)).cuda()
    y = torch.full_like(x, 7.0)
    engine.enqueue_prefill_route(model, b, 0, x, stacked=False, keep_logits=True)
    engine.enqueue_prefill_experts(model, b, 0, x, y, stacked=False, path=path)
    torch.cuda.synchronize()
    assert int(b.ctrl[1]) == 0
    xo = x.double().cpu().numpy()
    lg64 = oracle.router_logits(xo, o.router(0))
    rep = {}
    r = check_route(b.logits.cpu().numpy(), b.ids.cpu().numpy(), b.weights.cpu().numpy(), u64(b.slots), lg64,
                    o.table_row(0), w.top_k, 0, rep)
    assert rep.get("near_ties", 0) == 0
    offs, ptok, pk = oracle.build_pairs(r.ids, w.n_experts)
    assert np.array_equal(b.offs.cpu().numpy().astype(np.uint32), offs)
    P = T * w.top_k
    assert np.array_equal(b.pair_tok[:P].cpu().numpy().astype(np.uint32), ptok)
    assert np.array_equal(b.pair_k[:P].cpu().numpy(), pk)
    y_o = o.experts(xo, r.ids, r.weights, r.slots)
    tol = REL_F32 if path == "f32" else REL_TC
    assert rel_l2(y.cpu().numpy(), y_o) <= tol
