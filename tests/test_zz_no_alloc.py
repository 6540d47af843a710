"""moe_decode_static, the decode entry point for callers that cannot allocate device memory
(a plugin hosted by a program that owns every device allocation, a serving loop that forbids
allocation after start-up): its h scratch is a fixed array inside the library instead of a
caller workspace.  Two calls in a row must give what moe_decode gives with a workspace.
This file is collected last on purpose; it builds what it needs itself so it also passes
alone in a fresh process."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from tests._gpu_common import REL_F32, rel_l2  # noqa: E402


def test_static_scratch_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_moe_expert_rl_gb300 import _lib as L
    from quantized_moe_expert_rl_gb300 import build, engine
    build.build()
    w = synth.WORKLOADS["decode_layer"]
    m = engine.Model(w)
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w, 0, 2)).cuda()
    shp = m.shape
    for t in range(2):                          # two calls in a row, different routings
        L.rl_route(shp, 0, 1, x[t], -1.0, m.routers[0], None, m.table, b.ids[0], b.weights[0], b.slots[0], b.miss,
                   b.ctrl, None, b.route_ws, b.route_ws.numel())
        y_ws = torch.full((w.hidden,), 3.0, device="cuda")
        y_st = torch.full((w.hidden,), 3.0, device="cuda")
        L.moe_decode(shp, 0, x[t], -1.0, b.slots[0], b.weights[0], m.codebook, y_ws, 1, b.ctrl, b.dec_ws,
                     b.dec_ws.numel())
        L.moe_decode_static(shp, 0, x[t], -1.0, b.slots[0], b.weights[0], m.codebook, y_st, 1, b.ctrl)
        torch.cuda.synchronize()
        assert b.ctrl.tolist() == [0x7FFFFFFF, 0]
        a, r = y_st.double().cpu().numpy(), y_ws.double().cpu().numpy()
        assert rel_l2(a, r) <= REL_F32
        assert np.array_equal(a, r)            # the same kernels run; only the scratch differs
    # top_k * inter beyond the fixed scratch is refused before any launch.  Every supported
    # shape fits the array (the library asserts it at compile time), so the refusal comes from
    # the shape check that all entry points share.
    big = L.RlShape.of(2048, 512, 16, 2048, 1)
    with pytest.raises(L.RlError) as ei:
        L.moe_decode_static(big, 0, x[0], -1.0, b.slots[0], b.weights[0], m.codebook, x[1], 0, b.ctrl)
    assert ei.value.status == L.RL_ERR_UNSUPPORTED
    assert "top_k*inter" in str(ei.value)
