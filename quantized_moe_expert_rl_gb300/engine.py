"""Host-side drivers around the C ABI: the resident expert pool and residency table, the
per-token decode chain (captured as one CUDA graph per token), the prefill chunk chain, and
the bounded-residency chain with per-layer early-out, fill and resume.

PyTorch is used here only for device memory, pinned host memory, streams, events and
graphs.  Every step of the routed-MoE path runs in librlmoe's kernels.

Early-out and resume follow "Red Lite dev23 - per-layer early-out and pre-gated expert
prefetch", section "What changed", item 1: when layer f selects a non-resident expert the
router raises the flag, later kernels return at once, the host loads only layer f's missing
experts (here: copies their records from a pinned host backing store into free HBM slots and
updates the residency table), runs layer f with the ids and weights the GPU selected, and
resumes the chain at f + 1.  Nothing is evicted: the pool has a slot for every expert.
"""
from __future__ import annotations

import time
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _lib as L
from ._lib import RL_NO_EARLY_OUT, RlShape

EPS = 1e-6


def shape_of(w) -> RlShape:
    return RlShape.of(w.hidden, w.n_experts, w.top_k, w.inter, w.n_layers)


class Model:
    """A synthetic model resident on one GPU: codebook, routers (+ Zipf biases), the expert
    pool (one record slot per (layer, expert)), the residency table and, for bounded
    residency, a pinned host backing store of the absent experts' records."""

    def __init__(self, w, device="cuda", slot_perm: bool = False, layers: int | None = None,
                 gen_threads: int = 0):
        import synth
        self.w = w
        self.L = w.n_layers if layers is None else layers
        self.shape = RlShape.of(w.hidden, w.n_experts, w.top_k, w.inter, self.L)
        self.device = torch.device(device)
        E, H, rb = w.n_experts, w.hidden, w.record_bytes
        self.record_bytes = rb
        assert L.rl_record_bytes(self.shape) == rb
        self.codebook = torch.from_numpy(synth.grid(w.seed).reshape(-1).copy()).to(self.device)
        self.routers = torch.empty((self.L, E, H), dtype=torch.float32, device=self.device)
        self.bias = None
        if w.zipf_s > 0:
            self.bias = torch.empty((self.L, E), dtype=torch.float32, device=self.device)
        self.pool = torch.empty(self.L * E * rb, dtype=torch.uint8, device=self.device)
        base = self.pool.data_ptr()
        assert base % 256 == 0
        # slot position of each (layer, expert) inside the pool
        self.pos = np.empty((self.L, E), dtype=np.int64)
        for l in range(self.L):
            perm = synth.permutation(synth.TAG_SLOTPERM, l, E, w.seed) if slot_perm else np.arange(E)
            self.pos[l] = l * E + perm
        self.addr = (np.uint64(base) + self.pos.astype(np.uint64) * np.uint64(rb)).astype(np.uint64)
        self.resident = np.ones((self.L, E), dtype=bool)
        if w.n_resident >= 0:
            for l in range(self.L):
                self.resident[l] = synth.resident_mask(w, l).astype(bool)
        table = np.where(self.resident, self.addr, np.uint64(0)).astype(np.uint64)
        self.table_host = table.copy()
        self.table = torch.from_numpy(table.view(np.int64)).to(self.device)
        # upload: generate each layer into pinned staging, copy resident records to their slots
        stage = torch.empty((E, rb), dtype=torch.uint8, pin_memory=True)
        absent = [(l, e) for l in range(self.L) for e in range(E) if not self.resident[l, e]]
        self.backing = torch.empty((max(1, len(absent)), rb), dtype=torch.uint8, pin_memory=True)
        self.backing_index = {}
        stream = torch.cuda.current_stream(self.device)
        for l in range(self.L):
            stream.synchronize()
            synth.expert_records_into(stage.data_ptr(), w, l, 0, E, gen_threads)
            self.routers[l].copy_(torch.from_numpy(synth.router(w, l)))
            if self.bias is not None:
                self.bias[l].copy_(torch.from_numpy(synth.zipf_bias(w, l)))
            for e in range(E):
                if self.resident[l, e]:
                    p = int(self.pos[l, e])
                    self.pool[p * rb:(p + 1) * rb].copy_(stage[e], non_blocking=True)
                else:
                    j = len(self.backing_index)
                    self.backing[j].copy_(stage[e])
                    self.backing_index[(l, e)] = j
        stream.synchronize()
        del stage

    # -- helpers ------------------------------------------------------------------------
    def expert_of_addr(self) -> dict:
        """slot address -> (layer, expert), for checking slot tables."""
        return {int(self.addr[l, e]): (l, e) for l in range(self.L) for e in range(self.w.n_experts)}

    def record_host(self, layer: int, expert: int) -> np.ndarray:
        import synth
        return synth.expert_records(self.w, layer, expert, 1)[0]

    def fill(self, layer: int, experts, stream=None) -> int:
        """Copy the records of absent experts of `layer` from the pinned backing store into
        their free slots and mark them resident (host table and device table row).
        Returns the bytes copied."""
        rb = self.record_bytes
        s = stream or torch.cuda.current_stream(self.device)
        n = 0
        with torch.cuda.stream(s):
            for e in experts:
                if self.resident[layer, e]:
                    continue
                p = int(self.pos[layer, e])
                self.pool[p * rb:(p + 1) * rb].copy_(self.backing[self.backing_index[(layer, e)]], non_blocking=True)
                self.resident[layer, e] = True
                self.table_host[layer, e] = self.addr[layer, e]
                n += rb
            row = torch.from_numpy(self.table_host[layer].view(np.int64).copy()).pin_memory()
            self.table[layer].copy_(row, non_blocking=True)
        return n

    def device_fill_tables(self):
        """(src, dst) for rl_fill_missing: uint64 [L][E] device tensors holding, for every
        (layer, expert), the device-readable address of its record in the pinned backing store
        (0 when it has none) and the address of its HBM slot."""
        if getattr(self, "_fill_tables", None) is None:
            E, rb = self.w.n_experts, self.record_bytes
            src = np.zeros((self.L, E), dtype=np.uint64)
            if self.backing_index:
                base = L.rl_host_device_pointer(self.backing.data_ptr())
                for (l, e), j in self.backing_index.items():
                    src[l, e] = np.uint64(base + j * rb)
            self._fill_tables = (torch.from_numpy(src.view(np.int64)).to(self.device),
                                 torch.from_numpy(self.addr.view(np.int64).copy()).to(self.device))
        return self._fill_tables

    def sync_residency_from_device(self) -> None:
        """Bring the host mirror (table_host, resident) up to date after fills done by the
        device (rl_fill_missing)."""
        self.table_host = self.table.cpu().numpy().view(np.uint64).copy()
        self.resident = self.table_host != 0

    def reset_residency(self) -> None:
        """Forget fills: mark the seeded absent experts absent again (their slots keep
        whatever bytes they hold; the table no longer points at them)."""
        import synth
        if self.w.n_resident < 0:
            return
        for l in range(self.L):
            self.resident[l] = synth.resident_mask(self.w, l).astype(bool)
        self.table_host = np.where(self.resident, self.addr, np.uint64(0)).astype(np.uint64)
        self.table.copy_(torch.from_numpy(self.table_host.view(np.int64).copy()))


@dataclass
class DecodeBuffers:
    x: torch.Tensor          # [H] working residual stream of one token
    xn: torch.Tensor         # [H]
    ids: torch.Tensor        # [L][K] int32
    weights: torch.Tensor    # [L][K] f32
    slots: torch.Tensor      # [L][K] u64 (as int64)
    logits: torch.Tensor     # [L][E] f32
    miss: torch.Tensor       # [L] u32 (as int32)
    ctrl: torch.Tensor       # [2] int32
    route_ws: torch.Tensor
    dec_ws: torch.Tensor
    stack_ws: torch.Tensor   # zero-filled: grid-barrier counter of moe_decode_stack

    @staticmethod
    def make(model: Model) -> "DecodeBuffers":
        w, d = model.w, model.device
        Lh, K, E, H = model.L, w.top_k, w.n_experts, w.hidden
        shp = model.shape
        return DecodeBuffers(
            x=torch.zeros(H, dtype=torch.float32, device=d), xn=torch.zeros(H, dtype=torch.float32, device=d),
            ids=torch.zeros((Lh, K), dtype=torch.int32, device=d),
            weights=torch.zeros((Lh, K), dtype=torch.float32, device=d),
            slots=torch.zeros((Lh, K), dtype=torch.int64, device=d),
            logits=torch.zeros((Lh, E), dtype=torch.float32, device=d),
            miss=torch.zeros(Lh, dtype=torch.int32, device=d),
            ctrl=torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32, device=d),
            route_ws=torch.zeros(max(256, L.rl_route_workspace_bytes(shp, 1)), dtype=torch.uint8, device=d),
            dec_ws=torch.empty(L.moe_decode_workspace_bytes(shp), dtype=torch.uint8, device=d),
            stack_ws=torch.zeros(L.moe_decode_stack_workspace_bytes(shp), dtype=torch.uint8, device=d))


def enqueue_decode_token(model: Model, b: DecodeBuffers, x_in: torch.Tensor, y_out: torch.Tensor,
                         stacked: bool, keep_logits: bool = False, x_hist: torch.Tensor | None = None) -> None:
    """Enqueue one token through model.L layers on the current stream.

    stacked=False (one layer, no norm, no residual): y_out = MoE(x_in).
    stacked=True: x = x_in; per layer x = x + MoE(RMSNorm(x)) (the router and the experts
    normalise x on the fly); y_out = x.
    x_hist[l] (optional) receives layer l's input for per-layer checks."""
    shp = model.shape
    if not stacked:
        for l in range(model.L):
            L.rl_route(shp, l, 1, x_in, -1.0, model.routers[l], None if model.bias is None else model.bias[l],
                       model.table, b.ids[l], b.weights[l], b.slots[l], b.miss, b.ctrl,
                       b.logits[l] if keep_logits else None, b.route_ws, b.route_ws.numel())
            L.moe_decode(shp, l, x_in, -1.0, b.slots[l], b.weights[l], model.codebook, y_out, 0, b.ctrl, b.dec_ws,
                         b.dec_ws.numel())
        return
    b.x.copy_(x_in)
    for l in range(model.L):
        if x_hist is not None:
            x_hist[l].copy_(b.x)
        L.rl_route(shp, l, 1, b.x, EPS, model.routers[l], None if model.bias is None else model.bias[l],
                   model.table, b.ids[l], b.weights[l], b.slots[l], b.miss, b.ctrl,
                   b.logits[l] if keep_logits else None, b.route_ws, b.route_ws.numel())
        L.moe_decode(shp, l, b.x, EPS, b.slots[l], b.weights[l], model.codebook, b.x, 1, b.ctrl, b.dec_ws,
                     b.dec_ws.numel())
    y_out.copy_(b.x)


def enqueue_decode_layer_fused(model: Model, b: DecodeBuffers, x_in: torch.Tensor, y_out: torch.Tensor,
                               layer: int = 0, keep_logits: bool = False) -> None:
    """One token through one layer without norm or residual, router and experts in ONE launch
    (moe_decode_layer): y_out = MoE_layer(x_in), the same as enqueue_decode_token(stacked=False)
    for a one-layer model up to the order of the router's sums."""
    L.moe_decode_layer(model.shape, layer, x_in, -1.0, model.routers, model.bias, model.table, model.codebook,
                       b.ids, b.weights, b.slots, b.miss, b.ctrl, b.logits if keep_logits else None, y_out,
                       b.stack_ws, b.stack_ws.numel())


def enqueue_decode_token_fused(model: Model, b: DecodeBuffers, x_in: torch.Tensor, y_out: torch.Tensor,
                               keep_logits: bool = False, x_hist: torch.Tensor | None = None,
                               layer0: int = 0, pregate: int = 0,
                               pregate_hits: torch.Tensor | None = None) -> None:
    """Stacked decode of one token, layers [layer0, L), in ONE launch (moe_decode_stack):
    y_out = x_in, then per layer y_out += MoE(RMSNorm(y_out)).  The expert, RMSNorm and
    selection arithmetic is that of enqueue_decode_token(stacked=True); the router logits are
    summed across the launch's CTAs in 64-bit fixed point, so they agree with rl_route's to the
    last bits.  x_hist[l] (optional) receives layer l's input.
    pregate > 0 prefetches into L2 the next layer's predicted experts (never changes results);
    pregate_hits[l] (optional) receives how many of layer l's experts were predicted."""
    y_out.copy_(x_in)
    L.moe_decode_stack(model.shape, layer0, model.L - layer0, y_out, EPS, model.routers, model.bias, model.table,
                       model.codebook, b.ids, b.weights, b.slots, b.miss, b.ctrl, b.logits if keep_logits else None,
                       x_hist, pregate, pregate_hits, b.stack_ws, b.stack_ws.numel())


@dataclass
class DecodeStats:
    early_outs: list        # layers at which the chain stopped for a fill
    filled: list            # (layer, expert) filled at a stop
    fill_bytes: int
    syncs: int              # host reads of the control block or of routing results
    prefetched: list = field(default_factory=list)  # (layer, expert) filled ahead (lookahead)


def run_bounded_decode_token(model: Model, b: DecodeBuffers, x_in: torch.Tensor, y_out: torch.Tensor,
                             x_hist: torch.Tensor | None = None, pregate: int = 0,
                             lookahead: bool = False) -> DecodeStats:
    """One token through every layer with bounded residency ("Red Lite dev23", "What changed",
    item 1): the fused stack runs until a layer f selects an absent expert and stops there
    with y_out = x_f; the host reads the flag once, fills layer f's missing experts, re-resolves
    its slots, runs layer f's experts with the ids and weights the GPU selected, and restarts
    the stack at f + 1.  The caller zeroes b.miss; b.ctrl is reset here.

    lookahead: at each stop, before restarting, also route layer f+1 on x_{f+1} (known once
    layer f has run) and apply layer f+2's router to the same input (the pre-gated prediction
    of "Red Lite dev23 - per-layer early-out and pre-gated expert prefetch", "What changed":
    the next layer's router on this layer's input), and fill the absent experts of both, so
    that the restarted stack stops less often.  Results are unchanged; miss[l] then counts the
    misses the stack met after those fills."""
    shp, K = model.shape, model.w.top_k
    b.ctrl.copy_(torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32))
    y_out.copy_(x_in)
    st = DecodeStats([], [], 0, 0)
    scratch = None
    if lookahead:
        d = model.device
        scratch = dict(ids=torch.zeros((2, K), dtype=torch.int32, device=d),
                       weights=torch.zeros((2, K), dtype=torch.float32, device=d),
                       slots=torch.zeros((2, K), dtype=torch.int64, device=d),
                       miss=torch.zeros(model.L, dtype=torch.int32, device=d),
                       ctrl=torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32, device=d))
    l0 = 0
    while l0 < model.L:
        L.moe_decode_stack(shp, l0, model.L - l0, y_out, EPS, model.routers, model.bias, model.table,
                           model.codebook, b.ids, b.weights, b.slots, b.miss, b.ctrl, None, x_hist, pregate, None,
                           b.stack_ws, b.stack_ws.numel())
        ctrl = b.ctrl.tolist()
        st.syncs += 1
        if ctrl[1] != 0:
            raise RuntimeError(f"moe_decode_stack: device error bits {ctrl[1]:#x}")
        f = ctrl[0]
        if f == RL_NO_EARLY_OUT:
            break
        ids = b.ids[f].tolist()
        slots = b.slots[f].tolist()
        missing = sorted({ids[k] for k in range(K) if slots[k] == 0})
        st.fill_bytes += model.fill(f, missing)
        st.filled += [(f, e) for e in missing]
        st.early_outs.append(f)
        L.rl_resolve_slots(shp, f, 1, b.ids[f], model.table, b.slots[f])
        b.ctrl[0] = RL_NO_EARLY_OUT
        L.moe_decode(shp, f, y_out, EPS, b.slots[f], b.weights[f], model.codebook, y_out, 1, b.ctrl, b.dec_ws,
                     b.dec_ws.numel())
        if scratch is not None and f + 1 < model.L:
            # layer f+1 on x_{f+1} (exact but for summation order), layer f+2's router on the same
            # input (the pre-gated prediction); their absent experts are filled now
            ahead = [f + 1] + ([f + 2] if f + 2 < model.L else [])
            for j, la in enumerate(ahead):
                scratch["ctrl"].copy_(torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32))
                L.rl_route(shp, la, 1, y_out, EPS, model.routers[la], None if model.bias is None else model.bias[la],
                           model.table, scratch["ids"][j], scratch["weights"][j], scratch["slots"][j],
                           scratch["miss"], scratch["ctrl"], None, b.route_ws, b.route_ws.numel())
            pred = scratch["ids"][:len(ahead)].tolist()
            st.syncs += 1
            for la, row in zip(ahead, pred):
                absent = sorted({e for e in row if not model.resident[la, e]})
                st.fill_bytes += model.fill(la, absent)
                st.prefetched += [(la, e) for e in absent]
        l0 = f + 1
    return st


def run_bounded_decode_token_device(model: Model, b: DecodeBuffers, x_in: torch.Tensor, y_out: torch.Tensor,
                                    filled: torch.Tensor, x_hist: torch.Tensor | None = None) -> None:
    """One token through every layer with bounded residency in ONE launch: a layer that selects
    absent experts has them copied by the device from the pinned backing store into their slots
    and runs on (moe_decode_stack_fill); b.miss counts the misses per layer, `filled` (uint32
    [1], accumulated) the experts filled.  Same results as run_bounded_decode_token.  The caller
    zeroes b.miss; b.ctrl is reset here; call model.sync_residency_from_device() before using
    the host mirror of the table."""
    src, dst = model.device_fill_tables()
    b.ctrl.copy_(torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32))
    y_out.copy_(x_in)
    L.moe_decode_stack_fill(model.shape, 0, model.L, y_out, EPS, model.routers, model.bias, model.table,
                            model.codebook, b.ids, b.weights, b.slots, b.miss, b.ctrl, None, x_hist, src, dst, filled,
                            b.stack_ws, b.stack_ws.numel())


@dataclass
class PrefillBuffers:
    xn: torch.Tensor
    ids: torch.Tensor
    weights: torch.Tensor
    slots: torch.Tensor
    logits: torch.Tensor
    miss: torch.Tensor
    ctrl: torch.Tensor
    offs: torch.Tensor
    pair_tok: torch.Tensor
    pair_k: torch.Tensor
    route_ws: torch.Tensor
    ws: torch.Tensor
    fill_ws: torch.Tensor    # zero-filled: rl_fill_missing's claim flags and list
    fill_cnt: torch.Tensor   # [filled, first early-out] of device fills

    @staticmethod
    def make(model: Model, T: int) -> "PrefillBuffers":
        w, d, shp = model.w, model.device, model.shape
        K, E, H = w.top_k, w.n_experts, w.hidden
        return PrefillBuffers(
            xn=torch.zeros((T, H), dtype=torch.float32, device=d),
            ids=torch.zeros((T, K), dtype=torch.int32, device=d),
            weights=torch.zeros((T, K), dtype=torch.float32, device=d),
            slots=torch.zeros((T, K), dtype=torch.int64, device=d),
            logits=torch.zeros((T, E), dtype=torch.float32, device=d),
            miss=torch.zeros(model.L, dtype=torch.int32, device=d),
            ctrl=torch.tensor([RL_NO_EARLY_OUT, 0], dtype=torch.int32, device=d),
            offs=torch.zeros(E + 1, dtype=torch.int32, device=d),
            pair_tok=torch.zeros(max(1, T * K), dtype=torch.int32, device=d),
            pair_k=torch.zeros(max(1, T * K), dtype=torch.uint8, device=d),
            route_ws=torch.zeros(max(256, L.rl_route_workspace_bytes(shp, T)), dtype=torch.uint8, device=d),
            ws=torch.empty(max(256, L.moe_prefill_workspace_bytes(shp, T)), dtype=torch.uint8, device=d),
            fill_ws=torch.zeros(max(256, L.rl_fill_workspace_bytes(shp)), dtype=torch.uint8, device=d),
            fill_cnt=torch.tensor([0, RL_NO_EARLY_OUT], dtype=torch.int32, device=d))


def _experts_fn(path: str):
    return {"tc": L.moe_prefill_chunk, "f32": L.moe_prefill_chunk_f32}[path]


def enqueue_prefill_route(model: Model, b: PrefillBuffers, layer: int, x: torch.Tensor, stacked: bool,
                          keep_logits: bool = False) -> None:
    T, shp = x.shape[0], model.shape
    src = x
    if stacked:
        L.rl_rmsnorm(x, b.xn, T, model.w.hidden, EPS)
        src = b.xn
    L.rl_route(shp, layer, T, src, -1.0, model.routers[layer], None if model.bias is None else model.bias[layer],
               model.table, b.ids, b.weights, b.slots, b.miss, b.ctrl, b.logits if keep_logits else None,
               b.route_ws, b.route_ws.numel())


def enqueue_prefill_experts(model: Model, b: PrefillBuffers, layer: int, x: torch.Tensor, y: torch.Tensor,
                            stacked: bool, path: str = "tc") -> None:
    T, shp = x.shape[0], model.shape
    src = b.xn if stacked else x
    L.rl_build_pairs(shp, layer, T, b.ids, b.offs, b.pair_tok, b.pair_k, b.ctrl)
    _experts_fn(path)(shp, layer, T, src, b.offs, b.pair_tok, b.pair_k, b.slots, b.weights, model.codebook, y,
                      1 if stacked else 0, b.ctrl, b.ws, b.ws.numel())


@dataclass
class BoundedStats:
    miss: list
    first_early_out: int
    early_outs: list          # layers where the chain stopped
    filled: list              # (layer, expert) in fill order
    fill_bytes: int
    fill_seconds: float
    syncs: int


def run_bounded_chunk(model: Model, b: PrefillBuffers, x: torch.Tensor, path: str = "tc", window: int | None = None,
                      hist: dict | None = None) -> BoundedStats:
    """Prefill chunk through model.L stacked layers with bounded residency.

    The chain is enqueued `window` layers at a time; the host then reads the flag.  With
    window=None the window adapts: it starts at all layers, drops to one layer after an
    early-out (the next layers are likely to stop too, and every layer enqueued past a stop is
    a wasted launch) and doubles after each window that ran through.  If a layer f stopped the chain, its distinct missing experts
    are filled, its zero slots re-resolved, the flag reset, and the chain resumes with layer
    f's experts.  x is updated in place (x <- x + MoE(RMSNorm(x)) per layer).
    hist (optional): {"x": [L][T][H], "ids", "weights", "slots" ([L][T][K]), "logits" ([L][T][E])}
    device tensors that receive each layer's input and its routing as rl_route wrote it
    (slots before any fill)."""
    hist = hist or {}
    T, shp = x.shape[0], model.shape
    Lh = model.L
    adaptive = window is None
    window = Lh if window is None else window
    stats = BoundedStats([0] * Lh, RL_NO_EARLY_OUT, [], [], 0, 0.0, 0)
    b.miss.zero_()
    b.ctrl[0] = RL_NO_EARLY_OUT
    b.ctrl[1] = 0
    layer = 0
    resume_experts = False           # True: layer `layer` was routed already; run its experts
    while layer < Lh:
        end = min(Lh, layer + window)
        for l in range(layer, end):
            if not (resume_experts and l == layer):
                if "x" in hist:
                    hist["x"][l].copy_(x)
                enqueue_prefill_route(model, b, l, x, True, keep_logits="logits" in hist)
                for key, src in (("logits", b.logits), ("ids", b.ids), ("weights", b.weights), ("slots", b.slots)):
                    if key in hist:
                        hist[key][l].copy_(src)
            enqueue_prefill_experts(model, b, l, x, x, True, path)
        ctrl = b.ctrl.cpu()          # the host sync of the chain
        stats.syncs += 1
        if int(ctrl[1]) != 0:
            raise RuntimeError(f"device error bits {int(ctrl[1])} at layer {layer}")
        f = int(ctrl[0])
        if f == RL_NO_EARLY_OUT:
            layer = end
            resume_experts = False
            if adaptive:
                window = min(Lh, 2 * window)
            continue
        if adaptive:
            window = 1
        # layer f selected absent experts: fill, re-resolve, reset the flag, resume at f's experts
        t0 = time.perf_counter()
        ids = b.ids.cpu().numpy()
        slots = b.slots.cpu().numpy().view(np.uint64)
        missing = sorted(set(int(e) for e in ids[slots == 0]))
        nbytes = model.fill(f, missing)
        L.rl_resolve_slots(shp, f, T, b.ids, model.table, b.slots)
        b.ctrl[0] = RL_NO_EARLY_OUT
        torch.cuda.current_stream().synchronize()
        stats.fill_seconds += time.perf_counter() - t0
        stats.fill_bytes += nbytes
        stats.filled += [(f, e) for e in missing]
        stats.early_outs.append(f)
        if stats.first_early_out == RL_NO_EARLY_OUT:
            stats.first_early_out = f
        layer = f
        resume_experts = True
    stats.miss = [int(v) for v in b.miss.cpu().tolist()]
    return stats


def run_bounded_chunk_device(model: Model, b: PrefillBuffers, x: torch.Tensor, path: str = "tc",
                             hist: dict | None = None, timing: dict | None = None) -> BoundedStats:
    """Prefill chunk through model.L stacked layers with bounded residency and every fill done
    by the device: per layer rl_route (exact miss count, early-out flag), rl_fill_missing (the
    layer's absent selected experts copied from the pinned backing store into their slots, the
    slots re-resolved, the flag cleared), then the layer's experts, all enqueued at once with
    one host sync at the end.  Same selections, fills and outputs as run_bounded_chunk; the
    early-out layers are the layers that missed.  hist as for run_bounded_chunk.
    timing (optional, a dict): filled with the device time in ms of the three stages summed
    over the layers ("route": RMSNorm + rl_route, "fill": rl_fill_missing, "experts": pair
    build + grouped expert GEMMs), from CUDA events recorded on the current stream."""
    hist = hist or {}
    ev = [] if timing is not None else None

    def mark():
        if ev is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            ev.append(e)
    T, shp = x.shape[0], model.shape
    src, dst = model.device_fill_tables()
    table0 = model.table_host.copy()
    b.miss.zero_()
    b.ctrl[0] = RL_NO_EARLY_OUT
    b.ctrl[1] = 0
    b.fill_cnt[0] = 0
    b.fill_cnt[1] = RL_NO_EARLY_OUT
    filled, first = b.fill_cnt[0:1], b.fill_cnt[1:2]
    for l in range(model.L):
        if "x" in hist:
            hist["x"][l].copy_(x)
        mark()
        enqueue_prefill_route(model, b, l, x, True, keep_logits="logits" in hist)
        mark()
        for key, src_t in (("logits", b.logits), ("ids", b.ids), ("weights", b.weights), ("slots", b.slots)):
            if key in hist:
                hist[key][l].copy_(src_t)
        mark()
        L.rl_fill_missing(shp, l, T, b.ids, b.slots, model.table, src, dst, filled, first, b.ctrl, b.fill_ws,
                          b.fill_ws.numel())
        mark()
        enqueue_prefill_experts(model, b, l, x, x, True, path)
        mark()
    ctrl = b.ctrl.cpu()
    if ev is not None:
        torch.cuda.synchronize(model.device)
        t = {"route": 0.0, "fill": 0.0, "experts": 0.0}
        for l in range(model.L):
            e = ev[5 * l:5 * l + 5]
            t["route"] += e[0].elapsed_time(e[1])
            t["fill"] += e[2].elapsed_time(e[3])
            t["experts"] += e[3].elapsed_time(e[4])
        timing.update(t)
    if int(ctrl[1]) != 0:
        raise RuntimeError(f"device error bits {int(ctrl[1])} in a device-filled chunk")
    model.sync_residency_from_device()
    miss = [int(v) for v in b.miss.cpu().tolist()]
    cnt = b.fill_cnt.cpu().tolist()
    new = np.argwhere((table0 == 0) & (model.table_host != 0))
    fl = [(int(l), int(e)) for l, e in new]
    return BoundedStats(miss, int(cnt[1]), [l for l in range(model.L) if miss[l] > 0], fl,
                        int(cnt[0]) * model.record_bytes, 0.0, 1)
