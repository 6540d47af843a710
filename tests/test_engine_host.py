"""The host-side drivers of engine.py on the CPU, with the C library replaced by a stand-in
that follows the header's contract (tests/_fake_lib.py): the bounded-residency chunk (early-out,
fill of the missing experts, resume at the stopped layer's experts, the adaptive enqueue
window), the same chunk with the fills done by the device, and the bounded decode of one token
(stop, fill, moe_decode of the stopped layer, restart; with and without lookahead fills).

The drivers' bookkeeping (which layers stopped, which experts were filled and in what order,
the exact per-layer miss counts, the first early-out layer) is checked against the oracle's
stack recurrence with fills, and the outputs against the oracle from the driver's own layer
inputs.  Failures are made on the host: a fill source that raises, and device error bits
raised by a kernel stand-in."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from tests._fake_lib import FakeLib, FakeModel  # noqa: E402
from tests._gpu_common import rel_l2  # noqa: E402

# six layers of the small shape, 24 of 32 experts resident per layer, a Zipf-biased router
W = replace(synth.WORKLOADS["tiny"], n_layers=6, tokens=8, n_resident=24, zipf_s=1.1)


class _Stream:
    def synchronize(self):
        pass


@pytest.fixture
def host(monkeypatch):
    from quantized_moe_expert_rl_gb300 import engine
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a, **k: _Stream())

    def make(w=W):
        m = FakeModel(w)
        lib = FakeLib(m)
        lib.install(monkeypatch, engine)
        return engine, m, lib
    return make


def _oracle_stack(m, lib, x0, x_in):
    """The oracle's recurrence over every layer from the driver's own layer inputs, starting
    from the model's seeded residency (fills give each missing expert its slot)."""
    w = m.w
    layers = [oracle.LayerInputs(synth.router(w, l),
                                 np.where(synth.resident_mask(w, l).astype(bool), m.addr[l], np.uint64(0)),
                                 synth.zipf_bias(w, l) if w.zipf_s > 0 else None) for l in range(m.L)]
    return oracle.moe_stack(x0, layers, w.top_k, lib.record, w.hidden, w.inter, lib.grid,
                            new_slot=lambda l, e: int(m.addr[l, e]), x_in_override=x_in)


def _chunk(engine, m, window=None, device=False):
    x = torch.from_numpy(synth.tokens(m.w))
    x0 = x.clone()
    b = engine.PrefillBuffers.make(m, m.w.tokens)
    hist = {"x": torch.zeros((m.L, m.w.tokens, m.w.hidden))}
    if device:
        st = engine.run_bounded_chunk_device(m, b, x, hist=hist)
    else:
        st = engine.run_bounded_chunk(m, b, x, window=window, hist=hist)
    return st, x0, x, hist


def test_bounded_chunk_bookkeeping_matches_the_oracle(host):
    engine, m, lib = host()
    st, x0, x, hist = _chunk(engine, m)
    res = _oracle_stack(m, lib, x0.double().numpy(), [hist["x"][l].double().numpy() for l in range(m.L)])
    assert st.miss == res.miss and sum(res.miss) > 0
    assert st.first_early_out == res.first_early_out
    assert st.early_outs == [l for l in range(m.L) if res.miss[l] > 0]     # one stop per missing layer
    assert st.filled == res.fills                                           # same experts, same order
    assert st.fill_bytes == len(res.fills) * m.record_bytes
    assert rel_l2(x.double().numpy(), res.x_out) <= 1e-6
    assert np.array_equal(hist["x"][0].numpy(), x0.numpy())
    # every layer routed once, in order: after a fill the stopped layer runs with the ids and
    # weights already selected, it is not routed again
    assert [l for n, l in lib.runs if n == "rl_route"] == list(range(m.L))
    # the filled experts are resident afterwards, the others untouched
    for l, e in st.filled:
        assert m.resident[l, e] and m.table_host[l, e] == m.addr[l, e]
    assert int(m.resident.sum()) == m.L * W.n_resident + len(st.filled)


@pytest.mark.parametrize("window", [1, 2, W.n_layers])
def test_bounded_chunk_same_result_for_any_window(host, window):
    engine, m0, _ = host()
    ref, _, x_ref, _ = _chunk(engine, m0)
    engine, m, _ = host()
    st, _, x, _ = _chunk(engine, m, window=window)
    assert (st.miss, st.first_early_out, st.early_outs, st.filled) == \
           (ref.miss, ref.first_early_out, ref.early_outs, ref.filled)
    assert torch.equal(x, x_ref)
    assert len(st.early_outs) + 1 <= st.syncs <= 2 * m.L + 1


def test_device_fill_driver_equals_host_driver(host):
    engine, m0, _ = host()
    ref, _, x_ref, _ = _chunk(engine, m0)
    engine, m, lib = host()
    st, _, x, _ = _chunk(engine, m, device=True)
    assert st.miss == ref.miss and st.first_early_out == ref.first_early_out
    assert st.early_outs == ref.early_outs
    assert sorted(st.filled) == sorted(ref.filled)
    assert st.fill_bytes == ref.fill_bytes and st.syncs == 1
    assert torch.equal(x, x_ref)
    assert np.array_equal(m.table_host, m0.table_host)


def test_failing_fill_source_propagates_and_leaves_the_table(host):
    engine, m0, _ = host()
    ref, _, _, _ = _chunk(engine, m0)
    f = ref.early_outs[1]                      # the second layer that stops the chain
    engine, m, _ = host()
    table0 = m.table_host.copy()
    m.fail_fill_at = f
    with pytest.raises(OSError, match=f"layer {f}"):
        _chunk(engine, m)
    assert np.array_equal(m.table_host[f:], table0[f:])       # nothing filled from the failing layer on
    assert not np.array_equal(m.table_host[:f], table0[:f])   # the earlier stop was filled


def test_device_error_bits_stop_the_driver(host):
    engine, m, lib = host()
    lib.device_error_at = ("moe_prefill_chunk", 2)
    with pytest.raises(RuntimeError, match="device error bits"):
        _chunk(engine, m)


def _decode_tokens(engine, m, n, **kw):
    b = engine.DecodeBuffers.make(m)
    out, stats, hists = [], [], []
    for t in range(n):
        x = torch.from_numpy(synth.tokens(m.w, t, 1))[0]
        y = torch.zeros_like(x)
        hist = torch.zeros((m.L, m.w.hidden))
        b.miss.zero_()
        stats.append(engine.run_bounded_decode_token(m, b, x, y, x_hist=hist, **kw))
        out.append(y)
        hists.append(hist)
    return out, stats, hists, b


def test_bounded_decode_token_matches_the_oracle(host):
    engine, m, lib = host()
    table_start = m.table_host.copy()
    out, stats, hists, _ = _decode_tokens(engine, m, 3)
    filled_before = set()
    for t in range(3):
        x0 = synth.tokens(m.w, t, 1).astype(np.float64)
        layers = [oracle.LayerInputs(synth.router(W, l), table_start[l].copy(), synth.zipf_bias(W, l))
                  for l in range(m.L)]
        for l, e in filled_before:                 # residency only rises from token to token
            layers[l].table_row[e] = m.addr[l, e]
        res = oracle.moe_stack(x0, layers, W.top_k, lib.record, W.hidden, W.inter, lib.grid,
                               new_slot=lambda l, e: int(m.addr[l, e]),
                               x_in_override=[hists[t][l].double().numpy()[None] for l in range(m.L)])
        st = stats[t]
        assert st.early_outs == [l for l in range(m.L) if res.miss[l] > 0]
        assert st.filled == res.fills and st.fill_bytes == len(res.fills) * m.record_bytes
        # one flag read per launch: each stop, plus the run that reaches the last layer unless
        # the last stop was the last layer
        ends_on_stop = bool(st.early_outs) and st.early_outs[-1] == m.L - 1
        assert st.syncs == len(st.early_outs) + (0 if ends_on_stop else 1)
        assert rel_l2(out[t].double().numpy(), res.x_out[0]) <= 1e-6
        filled_before |= set(st.filled)
    assert sum(len(s.early_outs) for s in stats) > 0


def test_bounded_decode_lookahead_and_device_fill_agree(host):
    engine, m0, _ = host()
    ref, st0, _, _ = _decode_tokens(engine, m0, 3)
    engine, m1, _ = host()
    ahead, st1, _, _ = _decode_tokens(engine, m1, 3, lookahead=True)
    for a, r in zip(ahead, ref):
        assert torch.equal(a, r)
    stops0 = sum(len(s.early_outs) for s in st0)
    stops1 = sum(len(s.early_outs) for s in st1)
    assert stops1 <= stops0 and sum(len(s.prefetched) for s in st1) > 0
    # the fused stack with device fills: no stop at all, the same outputs and residency
    engine, m2, _ = host()
    b = engine.DecodeBuffers.make(m2)
    filled = torch.zeros(1, dtype=torch.int32)
    for t, r in enumerate(ref):
        x = torch.from_numpy(synth.tokens(m2.w, t, 1))[0]
        y = torch.zeros_like(x)
        engine.run_bounded_decode_token_device(m2, b, x, y, filled)
        assert torch.equal(y, r) and b.ctrl.tolist() == [0x7FFFFFFF, 0]
    m2.sync_residency_from_device()
    assert np.array_equal(m2.table_host, m0.table_host)
    assert int(filled[0]) == sum(len(s.filled) for s in st0)
