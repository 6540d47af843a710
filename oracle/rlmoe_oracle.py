"""Plain CPU oracle of the routed mixture-of-experts hot path.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline legs of `bench.py` may import this module.  The CUDA library never
calls it, shares no code with it, and the product path fails loudly instead of
falling back to it.

Everything is float64 unless a step is defined at another precision.  The code
is deliberately slow and literal: each function is the plain definition of one
step, with numpy library primitives (matmul, stable sort) as the only helpers.

Sources (the Red Lite engine notes):
  [dev21] "Red Lite dev21 - GPU-routed decode (full residency)", section
          "What changed": the layers x experts residency table (slot address,
          0 = not resident) and the rl_route kernel (softmax top-k by logit,
          ties to the lower index, weights renormalised over the selected
          experts, table lookups, slot table + weights + per-layer miss count).
  [dev23] "Red Lite dev23 - per-layer early-out and pre-gated expert prefetch",
          section "What changed", item 1: the early-out flag raised by rl_route
          at layer f, layers before f complete, layer f's misses loaded and run
          with the GPU's ids and weights, the chain resumed at f+1.
  [dev20] "Red Lite dev20 - batched prompt ingestion (native Metal prefill)",
          section "What changed", items 2-3: (expert, token) pairs sorted by
          expert, each token's top-k outputs accumulated in router selection
          order, union of a plan at most 512 experts.
  [dev38] "Red Lite dev38 - decode: expert down-projection lanes and concurrent
          encoders", section "Scope boundary": the order of the sums inside an
          expert's dot products is free; router ids must not change.
  [format] The synthetic 2.06-bpw codebook format of these workloads: a
          256-value block of 66 bytes = fp16 scale d, then 32 groups of 8
          values, each group a uint8 index into a 256 x 8 int8 grid plus a
          uint8 sign mask; value = d * grid[idx][j] * (+-1).  Expert output
          o = down(silu(gate x) * (up x)); layer output y = sum_k w_k o_k in
          selection order; stacks use x <- x + MoE(RMSNorm(x)), unit gain,
          eps 1e-6; bounded residency adds a Zipf router bias.

Readings where the sources are silent (the numbering is shared with the library's docs):
  R1 block bytes: d little-endian at bytes 0-1; group g at bytes 2+2g (idx)
     and 3+2g (sign); bit j of the sign byte (LSB = bit 0) negates value j.
  R2 a matrix is stored flat and row-major in consecutive 256-value blocks
     (so a 128-value row is half a block); an expert record is
     [gate I x H | up I x H | down H x I] back to back.
  R3 selection compares logits as real numbers (-0.0 == +0.0), descending,
     ties to the lower expert index; the selection is made on f32 logits
     (the router is an f32 GEMV) and the weights are computed in f64 from
     those f32 values: w_k = exp(l_k - l_1) / sum_j exp(l_j - l_1).
  R4 miss count = number of (token, k) selections whose slot is 0, with
     multiplicity; early_out = min over layers with a miss.
  R5 silu(z) = z / (1 + exp(-z)).
  R6 fill on early-out: each distinct missing expert of layer f gets a slot,
     table[f][e] is set, the zero slots are re-resolved, layer f's experts
     run, and the chain continues at f+1; nothing is evicted.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable

import numpy as np

BLOCK_VALUES = 256
BLOCK_BYTES = 66
NO_EARLY_OUT = 0x7FFFFFFF


# ----------------------------------------------------------------------------------------------
# Block format ([format], R1, R2)
# ----------------------------------------------------------------------------------------------
def fp16_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE 754 binary16 bit patterns -> float64, from the definition:
    sign bit 15, 5-bit exponent (bias 15) in bits 10-14, 10-bit fraction.
    Exponent 0 is subnormal (f/1024 * 2^-14); exponent 31 (inf/NaN) is rejected."""
    b = np.asarray(bits).astype(np.int64)
    sign = (b >> 15) & 1
    expo = (b >> 10) & 0x1F
    frac = b & 0x3FF
    if np.any(expo == 31):
        raise ValueError("fp16 inf/NaN scale in a block")
    normal = (1.0 + frac / 1024.0) * np.exp2(expo.astype(np.float64) - 15.0)
    subnormal = (frac / 1024.0) * 2.0 ** -14
    mag = np.where(expo == 0, subnormal, normal)
    return np.where(sign == 1, -mag, mag)


def dequantize(raw: np.ndarray, n_values: int, grid: np.ndarray) -> np.ndarray:
    """Decode consecutive 66-byte blocks into n_values float64 values (R1).

    value(block b, group g, j) = d_b * grid[idx_bg][j] * (-1 if bit j of sign_bg else +1)
    """
    raw = np.asarray(raw, dtype=np.uint8)
    nb = n_values // BLOCK_VALUES
    assert n_values % BLOCK_VALUES == 0 and raw.size >= nb * BLOCK_BYTES
    blocks = raw[: nb * BLOCK_BYTES].reshape(nb, BLOCK_BYTES)
    d = fp16_to_f64(blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8))
    idx = blocks[:, 2::2]                                  # [nb, 32] group index bytes
    sgn = blocks[:, 3::2]                                  # [nb, 32] group sign bytes
    mag = grid.astype(np.float64)[idx]                     # [nb, 32, 8]
    bit = (sgn[:, :, None].astype(np.int64) >> np.arange(8)) & 1
    vals = d[:, None, None] * mag * np.where(bit == 1, -1.0, 1.0)
    return vals.reshape(nb * BLOCK_VALUES)


def matrix_bytes(rows: int, cols: int) -> int:
    return rows * cols // BLOCK_VALUES * BLOCK_BYTES


def expert_weights(record: np.ndarray, hidden: int, inter: int, grid: np.ndarray):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) in float64 from one expert record (R2)."""
    mb = matrix_bytes(inter, hidden)
    record = np.asarray(record, dtype=np.uint8)
    wg = dequantize(record[0 * mb:1 * mb], inter * hidden, grid).reshape(inter, hidden)
    wu = dequantize(record[1 * mb:2 * mb], inter * hidden, grid).reshape(inter, hidden)
    wd = dequantize(record[2 * mb:3 * mb], hidden * inter, grid).reshape(hidden, inter)
    return wg, wu, wd


# ----------------------------------------------------------------------------------------------
# Router ([dev21] "What changed": rl_route; R3, R4)
# ----------------------------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Unit-gain RMSNorm of each row: x / sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def router_logits(xn: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """logits[t][e] = sum_h W_r[e][h] xn[t][h] (+ bias[e]), float64."""
    lg = np.asarray(xn, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    if bias is not None:
        lg = lg + np.asarray(bias, dtype=np.float64)[None, :]
    return lg


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """ids[t][0..k-1]: the k largest logits of each row in descending order, ties to the
    lower expert index; -0.0 and +0.0 are the same value (R3).  Uses numpy's stable lexsort
    on (negated value with -0 folded to +0, index)."""
    lg = np.atleast_2d(np.asarray(logits))
    if np.any(np.isnan(lg)):
        raise ValueError("NaN logit")
    neg = -lg + 0.0                                        # -(+0) = -0, and -0 + 0 = +0
    idx = np.broadcast_to(np.arange(lg.shape[1]), lg.shape)
    order = np.lexsort((idx, neg), axis=-1)                # primary: neg ascending; then index
    return order[:, :k].astype(np.int32)


def renorm_weights(logits: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """w[t][k] = exp(l_k - l_first) / sum_j exp(l_j - l_first) over the selected ids,
    float64, summed in selection order (R3).  Equals softmax-then-renormalise."""
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    e = np.exp(sel - sel[:, :1])
    total = np.zeros(sel.shape[0])
    for j in range(sel.shape[1]):
        total = total + e[:, j]
    return e / total[:, None]


def lookup(table_row: np.ndarray, ids: np.ndarray):
    """slots = table_row[ids] (uint64, 0 = not resident) and the miss count (R4)."""
    slots = np.asarray(table_row, dtype=np.uint64)[ids.astype(np.int64)]
    return slots, int(np.count_nonzero(slots == 0))


@dataclass
class RouteResult:
    ids: np.ndarray          # int32 [T][K], selection order
    weights: np.ndarray      # float64 [T][K]
    slots: np.ndarray        # uint64 [T][K]
    miss: int                # selections with slot 0
    early_out: int           # min(previous flag, layer) if miss else previous flag
    logits32: np.ndarray     # float32 [T][E]: the values the selection was made on


def route_from_logits(logits32: np.ndarray, table_row: np.ndarray, k: int, layer: int,
                      early_out: int = NO_EARLY_OUT) -> RouteResult:
    """Selection, weights, lookup, miss count and flag on given f32 logits."""
    lg = np.atleast_2d(np.asarray(logits32, dtype=np.float32))
    ids = select_topk(lg, k)
    w = renorm_weights(lg.astype(np.float64), ids)
    slots, miss = lookup(table_row, ids)
    flag = min(early_out, layer) if miss > 0 else early_out
    return RouteResult(ids, w, slots, miss, flag, lg)


def route(xn, w_router, bias, table_row, k: int, layer: int, early_out: int = NO_EARLY_OUT) -> RouteResult:
    """The whole router step: f64 logits rounded once to f32 (the router's precision),
    then route_from_logits."""
    lg32 = router_logits(xn, w_router, bias).astype(np.float32)
    return route_from_logits(lg32, table_row, k, layer, early_out)


# ----------------------------------------------------------------------------------------------
# Experts and the ordered sum ([format]; [dev20] "What changed" item 3; R5)
# ----------------------------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_forward(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, xn: np.ndarray) -> np.ndarray:
    """o = W_down (silu(W_gate xn) * (W_up xn)); xn may be one row [H] or rows [n][H]."""
    xn = np.asarray(xn, dtype=np.float64)
    g = xn @ wg.T
    u = xn @ wu.T
    h = silu(g) * u
    return h @ wd.T


def ordered_sum(outputs: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """y = w_0 o_0 + w_1 o_1 + ... accumulated strictly in selection order.
    outputs [T][K][H], weights [T][K] -> y [T][H]."""
    y = np.zeros((outputs.shape[0], outputs.shape[2]))
    for k in range(outputs.shape[1]):
        y = y + weights[:, k:k + 1] * outputs[:, k, :]
    return y


RecordSource = Callable[[int], np.ndarray]   # slot address -> expert record bytes


def moe_experts(xn: np.ndarray, ids: np.ndarray, weights: np.ndarray, slots: np.ndarray,
                records: RecordSource, hidden: int, inter: int, grid: np.ndarray) -> np.ndarray:
    """Routed-expert output y[t] = sum_k w[t][k] * expert(slot[t][k])(xn[t]), in k order.
    Every selected slot must be resident (non-zero).  Each distinct expert is decoded once."""
    xn = np.atleast_2d(np.asarray(xn, dtype=np.float64))
    T, K = ids.shape
    outs = np.zeros((T, K, hidden))
    for s in np.unique(slots):
        if int(s) == 0:
            raise ValueError("non-resident expert selected; fill it first")
        wg, wu, wd = expert_weights(records(int(s)), hidden, inter, grid)
        tt, kk = np.nonzero(slots == s)
        outs[tt, kk] = expert_forward(wg, wu, wd, xn[tt])
    return ordered_sum(outs, np.asarray(weights, dtype=np.float64))


# ----------------------------------------------------------------------------------------------
# Pairs sorted by expert ([dev20] "What changed" item 3)
# ----------------------------------------------------------------------------------------------
def build_pairs(ids: np.ndarray, n_experts: int):
    """Counting sort of the (token, k) selections by expert id, stable in (t, k) order.
    Returns offs [E+1] (uint32), pair_tok [T*K] (uint32), pair_k [T*K] (uint8)."""
    T, K = ids.shape
    key = ids.reshape(-1).astype(np.int64)                # flat index t*K + k
    order = np.argsort(key, kind="stable")
    counts = np.bincount(key, minlength=n_experts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    return offs, (order // K).astype(np.uint32), (order % K).astype(np.uint8)


def prefill_chunk(xn, ids, weights, slots, records, hidden, inter, grid, n_experts):
    """Batched chunk: per-pair outputs over the expert-sorted pairs, then each token's
    ordered sum.  Returns (y [T][H], pair_out [P][H] in pair order, offs, pair_tok, pair_k)."""
    xn = np.atleast_2d(np.asarray(xn, dtype=np.float64))
    T, K = ids.shape
    offs, ptok, pk = build_pairs(ids, n_experts)
    pair_out = np.zeros((T * K, hidden))
    for e in range(n_experts):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if lo == hi:
            continue
        s = int(slots[ptok[lo], pk[lo]])
        wg, wu, wd = expert_weights(records(s), hidden, inter, grid)
        pair_out[lo:hi] = expert_forward(wg, wu, wd, xn[ptok[lo:hi].astype(np.int64)])
    outs = np.zeros((T, K, hidden))
    outs[ptok.astype(np.int64), pk.astype(np.int64)] = pair_out
    return ordered_sum(outs, np.asarray(weights, dtype=np.float64)), pair_out, offs, ptok, pk


# ----------------------------------------------------------------------------------------------
# Stacks ([format] recurrence; [dev23] "What changed" item 1; R6)
# ----------------------------------------------------------------------------------------------
@dataclass
class LayerInputs:
    w_router: np.ndarray               # f32 [E][H]
    table_row: np.ndarray              # uint64 [E]
    bias: np.ndarray | None = None     # f32 [E]


@dataclass
class StackResult:
    x_out: np.ndarray
    x_in: list = field(default_factory=list)       # input of each layer
    routes: list = field(default_factory=list)     # RouteResult per layer (before any fill)
    miss: list = field(default_factory=list)
    first_early_out: int = NO_EARLY_OUT
    fills: list = field(default_factory=list)      # (layer, expert) filled, in fill order


def moe_stack(x0, layers: list[LayerInputs], k, records, hidden, inter, grid,
              eps: float = 1e-6, new_slot: Callable[[int, int], int] | None = None,
              x_in_override: list | None = None, first_layer: int = 0) -> StackResult:
    """x_{l+1} = x_l + MoE_l(RMSNorm(x_l)) over the given layers.

    If a layer selects a non-resident expert (miss > 0) the flag records the first such
    layer; then every distinct missing expert of that layer is given a slot by
    new_slot(layer, expert) (R6), the table row is updated, the slots are re-resolved and
    the layer completes.  x_in_override[l], if given, replaces the layer's input (teacher
    forcing of a per-layer comparison)."""
    x = np.atleast_2d(np.asarray(x0, dtype=np.float64))
    res = StackResult(x_out=x)
    flag = NO_EARLY_OUT
    for li, lay in enumerate(layers):
        layer = first_layer + li
        if x_in_override is not None and x_in_override[li] is not None:
            x = np.atleast_2d(np.asarray(x_in_override[li], dtype=np.float64))
        res.x_in.append(x)
        xn = rmsnorm(x, eps)
        r = route(xn, lay.w_router, lay.bias, lay.table_row, k, layer, flag)
        res.routes.append(r)
        res.miss.append(r.miss)
        flag = r.early_out
        slots = r.slots
        if r.miss > 0:
            if new_slot is None:
                raise ValueError(f"layer {layer}: {r.miss} misses and no fill source")
            for e in sorted(set(int(v) for v in r.ids[slots == 0])):
                lay.table_row[e] = np.uint64(new_slot(layer, e))
                res.fills.append((layer, e))
            slots, _ = lookup(lay.table_row, r.ids)
        y = moe_experts(xn, r.ids, r.weights, slots, records, hidden, inter, grid)
        x = x + y
    res.x_out = x
    res.first_early_out = flag
    return res
