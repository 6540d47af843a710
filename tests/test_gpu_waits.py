"""Bounded on-chip waits of the fused decode stack, made to run out on the GPU without any
fault: the test knobs in the workspace header shorten every wait of one launch and hold back
one CTA (it leaves before its first grid-barrier arrival, or it expects 16 bytes more than its
first router-column copy brings), so that the other CTAs' waits expire.  The launch must end
by itself with RL_DEVERR_WAIT_TIMEOUT in ctrl[1] and the early-out flag untouched; a launch on
the re-zeroed workspace then gives the bits of an undisturbed run.  Nothing traps and no wait
is unbounded: every wait of the kernel gives up after the given number of polls."""
from dataclasses import replace

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402

CAP = 4096          # polls per wait (a grid-barrier poll is an L2 round trip: a few ms in all)
KNOB_BYTE = 64      # u32 wait limit at byte 64, i32 hold-back selector at byte 68


def _engine():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_moe_expert_rl_gb300 import engine
    return engine


def _set_knobs(ws, cap, hold):
    ws.zero_()
    ws[KNOB_BYTE:KNOB_BYTE + 8].copy_(torch.tensor([cap, hold], dtype=torch.int32).view(torch.uint8))


@pytest.mark.parametrize("hold", [1, -1], ids=["cta0_never_arrives", "cta0_copy_short"])
def test_stack_wait_expiry(hold):
    engine = _engine()
    from quantized_moe_expert_rl_gb300 import _lib as L
    w = replace(synth.WORKLOADS["tiny"], n_layers=3)
    m = engine.Model(w)
    b = engine.DecodeBuffers.make(m)
    x = torch.from_numpy(synth.tokens(w, 0, 1)).cuda()[0]
    y_ref = torch.zeros(w.hidden, device="cuda")
    engine.enqueue_decode_token_fused(m, b, x, y_ref)
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [L.RL_NO_EARLY_OUT, 0]

    _set_knobs(b.stack_ws, CAP, hold)
    b.ctrl.copy_(torch.tensor([L.RL_NO_EARLY_OUT, 0], dtype=torch.int32))
    y = torch.zeros(w.hidden, device="cuda")
    engine.enqueue_decode_token_fused(m, b, x, y)
    torch.cuda.synchronize()                    # the launch ends by itself
    c = b.ctrl.tolist()
    assert c[0] == L.RL_NO_EARLY_OUT and c[1] & L.RL_DEVERR_WAIT_TIMEOUT, c

    # the counter is left mid-barrier: zero the workspace (knobs off), then an ordinary run
    b.stack_ws.zero_()
    b.ctrl.copy_(torch.tensor([L.RL_NO_EARLY_OUT, 0], dtype=torch.int32))
    y2 = torch.zeros(w.hidden, device="cuda")
    engine.enqueue_decode_token_fused(m, b, x, y2)
    torch.cuda.synchronize()
    assert b.ctrl.tolist() == [L.RL_NO_EARLY_OUT, 0]
    assert torch.equal(y2.view(torch.int32), y_ref.view(torch.int32))
    print(f"hold {hold}: ctrl after the held launch {c}; next launch bit-identical")
