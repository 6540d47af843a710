"""A host-only stand-in for the C library, for testing the Python drivers (engine.py) on the
CPU.  Each function follows what include/rl_moe.h states for the entry point of the same name
(the skip rules on ctrl[0], the miss count and flag, the fill of absent experts, the stop of
the fused stack at its first early-out layer), computes with the oracle on CPU tensors, and
can be told to fail.  It takes the place of the library's functions only inside tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from quantized_moe_expert_rl_gb300._lib import (RL_DEVERR_MISSING, RL_NO_EARLY_OUT, RlShape)


class FakeModel:
    """What the drivers read from engine.Model, on the CPU: routers, biases, the residency
    table (fake slot addresses), and fills that mark experts resident."""

    def __init__(self, w):
        self.w, self.L = w, w.n_layers
        self.shape = RlShape.of(w.hidden, w.n_experts, w.top_k, w.inter, w.n_layers)
        self.device = torch.device("cpu")
        self.record_bytes = w.record_bytes
        self.codebook = torch.from_numpy(synth.grid(w.seed).reshape(-1).copy())
        E = w.n_experts
        self.routers = torch.from_numpy(np.stack([synth.router(w, l) for l in range(self.L)]))
        self.bias = (torch.from_numpy(np.stack([synth.zipf_bias(w, l) for l in range(self.L)]))
                     if w.zipf_s > 0 else None)
        self.addr = ((np.arange(self.L * E, dtype=np.uint64).reshape(self.L, E) + np.uint64(1)) << np.uint64(12))
        self.resident = np.ones((self.L, E), dtype=bool)
        if w.n_resident >= 0:
            for l in range(self.L):
                self.resident[l] = synth.resident_mask(w, l).astype(bool)
        self.table_host = np.where(self.resident, self.addr, np.uint64(0)).astype(np.uint64)
        self.table = torch.from_numpy(self.table_host.view(np.int64).copy())
        self.fail_fill_at = None          # layer whose fill raises (a failing fill source)

    def expert_of(self, slot: int):
        i = (int(slot) >> 12) - 1
        return divmod(i, self.w.n_experts)

    def fill(self, layer, experts, stream=None) -> int:
        if layer == self.fail_fill_at:
            raise OSError(f"fill source failed at layer {layer}")
        n = 0
        for e in experts:
            if self.resident[layer, e]:
                continue
            self.resident[layer, e] = True
            self.table_host[layer, e] = self.addr[layer, e]
            n += self.record_bytes
        self.table[layer].copy_(torch.from_numpy(self.table_host[layer].view(np.int64).copy()))
        return n

    def device_fill_tables(self):
        src = np.where(self.resident, np.uint64(0), self.addr | np.uint64(1 << 40)).astype(np.uint64)
        return torch.from_numpy(src.view(np.int64).copy()), torch.from_numpy(self.addr.view(np.int64).copy())

    def sync_residency_from_device(self):
        self.table_host = self.table.numpy().view(np.uint64).copy()
        self.resident = self.table_host != 0


def _u64(t):
    return t.numpy().view(np.uint64)


class FakeLib:
    """Entry points of the library as the drivers call them (torch tensors, not pointers)."""

    def __init__(self, model: FakeModel):
        self.m = model
        self.w = model.w
        self.grid = synth.grid(model.w.seed)
        self.calls = []                   # every call: (name, layer)
        self.runs = []                    # the calls that did their work (not skipped on ctrl[0])
        self.device_error_at = None       # (function, layer): set a device error bit there
        self._rec = {}

    # -- helpers ---------------------------------------------------------------------------
    def record(self, slot):
        le = self.m.expert_of(slot)
        if le not in self._rec:
            self._rec[le] = synth.expert_records(self.w, le[0], le[1], 1)[0]
        return self._rec[le]

    def _xn(self, x, eps):
        x = x.double().numpy().reshape(-1, self.w.hidden)
        return oracle.rmsnorm(x, eps) if eps >= 0 else x

    def _route_into(self, layer, xn, w_router, bias, residency, ids, weights, slots, miss, ctrl, logits_out):
        lg = oracle.router_logits(xn, w_router.numpy(), None if bias is None else bias.numpy()).astype(np.float32)
        r = oracle.route_from_logits(lg, _u64(residency)[layer], self.w.top_k, layer)
        ids.view(-1)[:].copy_(torch.from_numpy(r.ids.reshape(-1)))
        weights.view(-1)[:].copy_(torch.from_numpy(r.weights.astype(np.float32).reshape(-1)))
        slots.view(-1)[:].copy_(torch.from_numpy(r.slots.view(np.int64).reshape(-1)))
        if logits_out is not None:
            logits_out.view(-1)[:].copy_(torch.from_numpy(lg.reshape(-1)))
        miss[layer] += r.miss
        if r.miss > 0:
            ctrl[0] = min(int(ctrl[0]), layer)
        return r

    def _experts(self, xn, slots_np, weights_np):
        ids = np.zeros(slots_np.shape, dtype=np.int32)
        return oracle.moe_experts(xn, ids, weights_np, slots_np, self.record, self.w.hidden, self.w.inter, self.grid)

    def _dev_error(self, fn, layer, ctrl):
        if self.device_error_at == (fn, layer):
            ctrl[1] = int(ctrl[1]) | RL_DEVERR_MISSING

    # -- workspace queries -------------------------------------------------------------------
    def rl_route_workspace_bytes(self, shape, T):
        return 256

    def moe_decode_workspace_bytes(self, shape):
        return 256

    def moe_decode_stack_workspace_bytes(self, shape):
        return 256

    def moe_prefill_workspace_bytes(self, shape, T):
        return 256

    def rl_fill_workspace_bytes(self, shape):
        return 256

    # -- entry points ------------------------------------------------------------------------
    def rl_rmsnorm(self, x, xn, T, H, eps, stream=None):
        self.calls.append(("rl_rmsnorm", None))
        if T:
            xn[:T].copy_(torch.from_numpy(oracle.rmsnorm(x[:T].double().numpy(), eps).astype(np.float32)))

    def rl_route(self, shape, layer, T, x, norm_eps, w_router, bias, residency, ids, weights, slots, miss, ctrl,
                 logits_out=None, ws=None, ws_bytes=0, stream=None):
        self.calls.append(("rl_route", layer))
        if T == 0 or int(ctrl[0]) < layer:
            return
        self.runs.append(("rl_route", layer))
        self._route_into(layer, self._xn(x[:T] if x.dim() > 1 else x, norm_eps), w_router, bias, residency, ids,
                         weights, slots, miss, ctrl, logits_out)

    def rl_resolve_slots(self, shape, layer, T, ids, residency, slots, stream=None):
        self.calls.append(("rl_resolve_slots", layer))
        row = _u64(residency)[layer]
        slots.view(-1)[:].copy_(torch.from_numpy(row[ids.view(-1).numpy().astype(np.int64)].view(np.int64)))

    def rl_build_pairs(self, shape, layer, T, ids, offs, pair_tok, pair_k, ctrl, ws=None, ws_bytes=0, stream=None):
        self.calls.append(("rl_build_pairs", layer))
        if int(ctrl[0]) <= layer:
            return
        o, pt, pk = oracle.build_pairs(ids[:T].numpy(), self.w.n_experts)
        offs.copy_(torch.from_numpy(o.astype(np.int32)))
        pair_tok[:len(pt)].copy_(torch.from_numpy(pt.astype(np.int32)))
        pair_k[:len(pk)].copy_(torch.from_numpy(pk))

    def _prefill(self, name, shape, layer, T, xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate,
                 ctrl, ws, ws_bytes, stream=None):
        self.calls.append((name, layer))
        if int(ctrl[0]) <= layer:
            return
        self._dev_error(name, layer, ctrl)
        sl = _u64(slots[:T])
        if np.any(sl == 0):
            ctrl[1] = int(ctrl[1]) | RL_DEVERR_MISSING
            return
        out = self._experts(xn[:T].double().numpy(), sl, weights[:T].double().numpy())
        base = y[:T].double().numpy() if accumulate else 0.0
        y[:T].copy_(torch.from_numpy((base + out).astype(np.float32)))

    def moe_prefill_chunk(self, *a, **k):
        self._prefill("moe_prefill_chunk", *a, **k)

    def moe_prefill_chunk_f32(self, *a, **k):
        self._prefill("moe_prefill_chunk_f32", *a, **k)

    def rl_fill_missing(self, shape, layer, T, ids, slots, residency, src, dst, filled, first_early_out, ctrl, ws,
                        ws_bytes, stream=None):
        self.calls.append(("rl_fill_missing", layer))
        table = residency.numpy().view(np.uint64)
        sl = _u64(slots[:T]).reshape(-1)
        idv = ids[:T].numpy().reshape(-1)
        need = sorted({int(e) for e, s in zip(idv, sl) if s == 0})
        for e in need:
            if int(src[layer, e]) == 0 or int(dst[layer, e]) == 0:
                ctrl[1] = int(ctrl[1]) | RL_DEVERR_MISSING
                continue
            table[layer, e] = np.uint64(int(dst[layer, e]))
            filled[0] += 1
        if need:
            first_early_out[0] = min(int(first_early_out[0]), layer)
            if int(ctrl[0]) == layer:
                ctrl[0] = RL_NO_EARLY_OUT
        self.rl_resolve_slots(shape, layer, T, ids[:T], residency, slots[:T])

    def moe_decode(self, shape, layer, x, norm_eps, slots, weights, codebook, y, accumulate, ctrl, ws, ws_bytes,
                   stream=None):
        self.calls.append(("moe_decode", layer))
        if int(ctrl[0]) <= layer:
            return
        sl = _u64(slots).reshape(1, -1)
        if np.any(sl == 0):
            ctrl[1] = int(ctrl[1]) | RL_DEVERR_MISSING
            return
        out = self._experts(self._xn(x, norm_eps), sl, weights.double().numpy().reshape(1, -1))[0]
        base = y.double().numpy() if accumulate else 0.0
        y.copy_(torch.from_numpy((base + out).astype(np.float32)))

    def _stack(self, name, shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids, weights,
               slots, miss, ctrl, logits_out, x_hist, fill=None):
        self.calls.append((name, layer0))
        if int(ctrl[0]) < layer0:
            return
        for l in range(layer0, layer0 + n_layers):
            if x_hist is not None:
                x_hist[l].copy_(x)
            xn = self._xn(x, norm_eps)
            r = self._route_into(l, xn, w_router[l], None if bias is None else bias[l], residency, ids[l],
                                 weights[l], slots[l], miss, ctrl, None if logits_out is None else logits_out[l])
            if r.miss > 0:
                if fill is None:
                    return                      # stop: x stays the input of layer l
                src, dst, filled = fill
                self.rl_fill_missing(shape, l, 1, ids[l:l + 1], slots[l:l + 1], residency, src, dst, filled,
                                     torch.tensor([RL_NO_EARLY_OUT], dtype=torch.int32), ctrl, None, 0)
            self._dev_error(name, l, ctrl)
            sl = _u64(slots[l]).reshape(1, -1)
            out = self._experts(xn, sl, weights[l].double().numpy().reshape(1, -1))[0]
            x.copy_(torch.from_numpy((x.double().numpy() + out).astype(np.float32)))

    def moe_decode_stack(self, shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids,
                         weights, slots, miss, ctrl, logits_out, x_hist, pregate, pregate_hits, ws, ws_bytes,
                         stream=None):
        self._stack("moe_decode_stack", shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook,
                    ids, weights, slots, miss, ctrl, logits_out, x_hist)

    def moe_decode_stack_fill(self, shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids,
                              weights, slots, miss, ctrl, logits_out, x_hist, fill_src, fill_dst, filled, ws,
                              ws_bytes, stream=None):
        self._stack("moe_decode_stack_fill", shape, layer0, n_layers, x, norm_eps, w_router, bias, residency,
                    codebook, ids, weights, slots, miss, ctrl, logits_out, x_hist, fill=(fill_src, fill_dst, filled))

    NAMES = ("rl_route_workspace_bytes", "moe_decode_workspace_bytes", "moe_decode_stack_workspace_bytes",
             "moe_prefill_workspace_bytes", "rl_fill_workspace_bytes", "rl_rmsnorm", "rl_route", "rl_resolve_slots",
             "rl_build_pairs", "moe_prefill_chunk", "moe_prefill_chunk_f32", "rl_fill_missing", "moe_decode",
             "moe_decode_stack", "moe_decode_stack_fill")

    def install(self, monkeypatch, engine):
        for n in self.NAMES:
            monkeypatch.setattr(engine.L, n, getattr(self, n))
