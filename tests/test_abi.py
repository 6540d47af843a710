"""The C-ABI library: it loads, exports every symbol include/rl_moe.h declares, and answers
the host-only queries (no kernel launch, no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_moe_expert_rl_gb300 import _lib, build
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "rl_moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"sizeof"})


def test_exports_every_declared_symbol(lib):
    from quantized_moe_expert_rl_gb300 import _lib
    declared = _declared()
    assert set(declared) == set(_lib.EXPORTS), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_host_queries(lib):
    from quantized_moe_expert_rl_gb300._lib import RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    assert lib.rl_abi_version() == 1
    assert lib.rl_record_bytes(ctypes.byref(s)) == 811008
    assert lib.moe_decode_workspace_bytes(ctypes.byref(s)) >= 10 * 512 * 4
    assert lib.rl_route_workspace_bytes(ctypes.byref(s), 2048) >= 2048 * 512 * 4
    assert lib.moe_prefill_workspace_bytes(ctypes.byref(s), 512) >= 5120 * 512 * 4 + 5120 * 2048 * 4
    assert lib.rl_record_bytes(None) == 0


def test_invalid_arguments_are_rejected_before_launch(lib):
    """Checks that fail on the host: they return a status and launch nothing, so they run
    without a GPU."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RL_ERR_UNSUPPORTED, RlShape
    good = RlShape.of(2048, 512, 10, 512, 48)
    fake = ctypes.c_void_p(1 << 20)
    # layer out of range
    st = lib.rl_route(ctypes.byref(good), 48, 1, fake, -1.0, fake, None, fake, fake, fake, fake, fake, fake, fake, None,
                      0, None)
    assert st == RL_ERR_INVALID and b"layer" in lib.rl_last_error()
    # NULL required buffer
    st = lib.moe_decode(ctypes.byref(good), 0, None, -1.0, fake, fake, fake, fake, 0, fake, fake, 1 << 20, None)
    assert st == RL_ERR_INVALID
    # workspace too small
    st = lib.moe_decode(ctypes.byref(good), 0, fake, -1.0, fake, fake, fake, fake, 0, fake, fake, 16, None)
    assert st == RL_ERR_INVALID and b"workspace" in lib.rl_last_error()
    # unsupported shapes
    for bad in (RlShape.of(384, 512, 10, 512, 1), RlShape.of(2048, 1024, 10, 512, 1),
                RlShape.of(2048, 512, 17, 512, 1), RlShape.of(2048, 512, 10, 200, 1)):
        st = lib.rl_build_pairs(ctypes.byref(bad), 0, 4, fake, fake, fake, fake, fake, None, 0, None)
        assert st == RL_ERR_UNSUPPORTED, bad
    # top_k > n_experts
    st = lib.rl_build_pairs(ctypes.byref(RlShape.of(512, 8, 10, 128, 1)), 0, 4, fake, fake, fake, fake, fake, None,
                            0, None)
    assert st == RL_ERR_INVALID
    # prefill workspace too small / misaligned
    st = lib.moe_prefill_chunk(ctypes.byref(good), 0, 512, fake, fake, fake, fake, fake, fake, fake, fake, 0, fake,
                               fake, 1024, None)
    assert st == RL_ERR_INVALID
    st = lib.rl_rmsnorm(fake, fake, 4, 2048, -1.0, None)
    assert st == RL_ERR_INVALID


def test_decode_stack_host_checks(lib):
    """moe_decode_stack: workspace query and the checks made before any launch."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RL_OK, RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    need = lib.moe_decode_stack_workspace_bytes(ctypes.byref(s))
    assert need >= 256 + 512 * 4 + 10 * 512 * 4
    fake = ctypes.c_void_p(1 << 20)
    args = [fake, -1.0, fake, None, fake, fake, fake, fake, fake, fake, fake, None, None, 0, None, fake]
    # layers outside [0, n_layers)
    assert lib.moe_decode_stack(ctypes.byref(s), 40, 9, *args, need, None) == RL_ERR_INVALID
    assert b"layers" in lib.rl_last_error()
    # workspace too small
    assert lib.moe_decode_stack(ctypes.byref(s), 0, 48, *args, need - 256, None) == RL_ERR_INVALID
    assert b"workspace" in lib.rl_last_error()
    # NULL required buffer (x)
    bad = list(args)
    bad[0] = None
    assert lib.moe_decode_stack(ctypes.byref(s), 0, 48, *bad, need, None) == RL_ERR_INVALID
    # misaligned router weights
    bad = list(args)
    bad[2] = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_decode_stack(ctypes.byref(s), 0, 48, *bad, need, None) == RL_ERR_INVALID
    # pregate beyond the 32 experts it can prefetch
    bad = list(args)
    bad[13] = 33
    assert lib.moe_decode_stack(ctypes.byref(s), 0, 48, *bad, need, None) == RL_ERR_INVALID
    # zero layers: nothing to do, no launch
    assert lib.moe_decode_stack(ctypes.byref(s), 48, 0, *args, need, None) == RL_OK


def test_decode_layer_host_checks(lib):
    """moe_decode_layer: the checks made before any launch (NULL y, layer out of range,
    workspace too small, misaligned x)."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RlShape
    s = RlShape.of(2048, 512, 10, 512, 1)
    need = lib.moe_decode_stack_workspace_bytes(ctypes.byref(s))
    fake = ctypes.c_void_p(1 << 20)
    # x, eps, router, bias, table, codebook, ids, weights, slots, miss, ctrl, logits, y
    args = [fake, -1.0, fake, None, fake, fake, fake, fake, fake, fake, fake, None, fake]
    bad = list(args)
    bad[12] = None
    assert lib.moe_decode_layer(ctypes.byref(s), 0, *bad, fake, need, None) == RL_ERR_INVALID
    assert b"NULL y" in lib.rl_last_error()
    assert lib.moe_decode_layer(ctypes.byref(s), 1, *args, fake, need, None) == RL_ERR_INVALID
    assert lib.moe_decode_layer(ctypes.byref(s), 0, *args, fake, need - 256, None) == RL_ERR_INVALID
    bad = list(args)
    bad[0] = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_decode_layer(ctypes.byref(s), 0, *bad, fake, need, None) == RL_ERR_INVALID


def test_fill_host_checks(lib):
    """rl_fill_missing, moe_decode_stack_fill and rl_host_device_pointer: the checks made
    before any launch (no GPU needed)."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    need = lib.rl_fill_workspace_bytes(ctypes.byref(s))
    assert need >= 512 * 8
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 8   # ids, slots, residency, src, dst, filled, first_early_out, ctrl
    assert lib.rl_fill_missing(ctypes.byref(s), 48, 4, *args, fake, need, None) == RL_ERR_INVALID
    assert b"layer" in lib.rl_last_error()
    assert lib.rl_fill_missing(ctypes.byref(s), 0, 4, *args, fake, need - 8, None) == RL_ERR_INVALID
    assert b"workspace" in lib.rl_last_error()
    bad = list(args)
    bad[3] = None
    assert lib.rl_fill_missing(ctypes.byref(s), 0, 4, *bad, fake, need, None) == RL_ERR_INVALID
    # the fused decode with fills needs its fill tables
    need_st = lib.moe_decode_stack_workspace_bytes(ctypes.byref(s))
    st_args = [fake, -1.0, fake, None, fake, fake, fake, fake, fake, fake, fake, None, None]
    assert lib.moe_decode_stack_fill(ctypes.byref(s), 0, 48, *st_args, None, fake, fake, fake, need_st,
                                     None) == RL_ERR_INVALID
    assert b"fill" in lib.rl_last_error()
    # a pointer that is not page-locked host memory has no device address
    out = ctypes.c_uint64(0)
    buf = ctypes.create_string_buffer(64)
    assert lib.rl_host_device_pointer(ctypes.cast(buf, ctypes.c_void_p), ctypes.byref(out)) == RL_ERR_INVALID
    assert lib.rl_host_device_pointer(None, ctypes.byref(out)) == RL_ERR_INVALID


def test_binding_refuses_strided_and_host_tensors():
    """The binding passes raw addresses; a view with gaps or a host tensor would be read as
    something else by the kernels, so it is refused before any call."""
    torch = pytest.importorskip("torch")
    from quantized_moe_expert_rl_gb300._lib import ptr
    assert ptr(None) is None and ptr(0) is None and ptr(4096) == 4096
    with pytest.raises(ValueError, match="contiguous"):
        ptr(torch.zeros(4, 4)[:, 1])
    with pytest.raises(ValueError, match="device buffer"):
        ptr(torch.zeros(4))


def test_zero_tokens_is_a_no_op(lib):
    """T = 0: rl_route, rl_rmsnorm, rl_resolve_slots and the prefill chunk return RL_OK
    without a launch and without reading their per-token buffers (NULL here); a bad layer or
    a negative T is still refused."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RL_OK, RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    fake = ctypes.c_void_p(1 << 20)
    n = [None] * 9
    assert lib.rl_route(ctypes.byref(s), 3, 0, None, -1.0, *n, None, 0, None) == RL_OK
    assert lib.rl_route(ctypes.byref(s), 48, 0, None, -1.0, *n, None, 0, None) == RL_ERR_INVALID
    assert lib.rl_route(ctypes.byref(s), 3, -1, None, -1.0, *n, None, 0, None) == RL_ERR_INVALID
    assert lib.rl_rmsnorm(None, None, 0, 2048, 1e-6, None) == RL_OK
    assert lib.rl_rmsnorm(None, None, 1, 2048, 1e-6, None) == RL_ERR_INVALID
    assert lib.rl_resolve_slots(ctypes.byref(s), 3, 0, None, None, None, None) == RL_OK
    for fn in (lib.moe_prefill_chunk, lib.moe_prefill_chunk_f32):
        assert fn(ctypes.byref(s), 3, 0, None, fake, None, None, None, None, None, None, 0, fake, None, 0,
                  None) == RL_OK


def test_selection_counts_beyond_the_index_range_are_refused(lib):
    """T * top_k above 2^30 selections would overflow the kernels' 32-bit pair indices: every
    entry point that takes T refuses it on the host."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_UNSUPPORTED, RlShape
    s = RlShape.of(2048, 512, 16, 512, 48)
    T = (1 << 26) + 1                          # 16 * T > 2^30
    fake = ctypes.c_void_p(1 << 20)
    ws = lib.rl_route_workspace_bytes(ctypes.byref(s), T)
    assert lib.rl_route(ctypes.byref(s), 0, T, fake, -1.0, fake, None, fake, fake, fake, fake, fake, fake, None,
                        fake, ws, None) == RL_ERR_UNSUPPORTED
    assert lib.rl_resolve_slots(ctypes.byref(s), 0, T, fake, fake, fake, None) == RL_ERR_UNSUPPORTED
    assert lib.rl_build_pairs(ctypes.byref(s), 0, T, fake, fake, fake, fake, fake, None, 0, None) == RL_ERR_UNSUPPORTED
    need = lib.rl_fill_workspace_bytes(ctypes.byref(s))
    assert lib.rl_fill_missing(ctypes.byref(s), 0, T, *([fake] * 8), fake, need, None) == RL_ERR_UNSUPPORTED
    for fn in (lib.moe_prefill_chunk, lib.moe_prefill_chunk_f32):
        assert fn(ctypes.byref(s), 0, T, *([fake] * 7), fake, 0, fake, fake, 1 << 62, None) == RL_ERR_UNSUPPORTED


def test_prefill_host_checks(lib):
    """moe_prefill_chunk and moe_prefill_chunk_f32: a layer out of range, a NULL per-token
    buffer, a workspace too small and xn, y or ws off a 16-byte boundary are refused before any
    launch (no GPU needed), with the reason in rl_last_error."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    T = 512
    need = lib.moe_prefill_workspace_bytes(ctypes.byref(s), T)
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)

    def args(xn=fake, y=fake, ws=fake, ws_bytes=need, weights=fake):
        # xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate, ctrl, ws, ws_bytes
        return [xn, fake, fake, fake, fake, weights, fake, y, 0, fake, ws, ws_bytes, None]
    for fn in (lib.moe_prefill_chunk, lib.moe_prefill_chunk_f32):
        assert fn(ctypes.byref(s), 48, T, *args()) == RL_ERR_INVALID
        assert b"layer" in lib.rl_last_error()
        assert fn(ctypes.byref(s), -1, T, *args()) == RL_ERR_INVALID
        assert fn(ctypes.byref(s), 0, -1, *args()) == RL_ERR_INVALID
        assert fn(ctypes.byref(s), 0, T, *args(weights=None)) == RL_ERR_INVALID
        assert b"NULL" in lib.rl_last_error()
        assert fn(ctypes.byref(s), 0, T, *args(ws_bytes=need - 16)) == RL_ERR_INVALID
        assert b"workspace" in lib.rl_last_error()
        for bad in (dict(xn=odd), dict(y=odd), dict(ws=odd)):
            assert fn(ctypes.byref(s), 0, T, *args(**bad)) == RL_ERR_INVALID, bad
            assert b"aligned" in lib.rl_last_error()


def test_pairs_and_slots_host_checks(lib):
    """rl_build_pairs and rl_resolve_slots: a layer out of range, a negative T and a NULL
    buffer are refused before any launch (no GPU needed)."""
    from quantized_moe_expert_rl_gb300._lib import RL_ERR_INVALID, RlShape
    s = RlShape.of(2048, 512, 10, 512, 48)
    fake = ctypes.c_void_p(1 << 20)
    # ids, offs, pair_tok, pair_k, ctrl
    good = [fake] * 5
    assert lib.rl_build_pairs(ctypes.byref(s), 48, 4, *good, None, 0, None) == RL_ERR_INVALID
    assert b"layer" in lib.rl_last_error()
    assert lib.rl_build_pairs(ctypes.byref(s), 0, -1, *good, None, 0, None) == RL_ERR_INVALID
    for i in range(5):
        bad = list(good)
        bad[i] = None
        assert lib.rl_build_pairs(ctypes.byref(s), 0, 4, *bad, None, 0, None) == RL_ERR_INVALID, i
    # with no selections the per-selection buffers may be NULL, offs and ctrl may not
    assert lib.rl_build_pairs(ctypes.byref(s), 0, 0, None, None, None, None, fake, None, 0, None) == RL_ERR_INVALID
    assert lib.rl_build_pairs(ctypes.byref(s), 0, 0, None, fake, None, None, None, None, 0, None) == RL_ERR_INVALID
    # ids, residency, slots
    assert lib.rl_resolve_slots(ctypes.byref(s), 48, 4, fake, fake, fake, None) == RL_ERR_INVALID
    assert lib.rl_resolve_slots(ctypes.byref(s), 0, -1, fake, fake, fake, None) == RL_ERR_INVALID
    for i in range(3):
        bad = [fake] * 3
        bad[i] = None
        assert lib.rl_resolve_slots(ctypes.byref(s), 0, 4, *bad, None) == RL_ERR_INVALID, i
