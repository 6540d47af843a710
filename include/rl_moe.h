/*
 * rl_moe.h - C ABI of the routed mixture-of-experts hot path on GB300 (sm_103a).
 *
 * The path, as the Red Lite engine notes describe it:
 *   router  : f32 GEMV to expert logits, softmax top-k (candidates ordered by
 *             logit, ties to the lower expert index), weights renormalised over
 *             the selected experts, lookup of each selected expert in a
 *             layers x experts residency table (slot address, 0 = absent), a
 *             per-layer miss count and an early-out flag
 *             ("Red Lite dev21 - GPU-routed decode (full residency)", section
 *             "What changed": residency table, rl_route kernel;
 *             "Red Lite dev23 - per-layer early-out and pre-gated expert
 *             prefetch", section "What changed", item 1);
 *   experts : gate/up/down projections of quantized experts with SwiGLU;
 *   combine : each token's top-k outputs weighted and summed in router
 *             selection order
 *             ("Red Lite dev20 - batched prompt ingestion (native Metal
 *             prefill)", section "What changed", items 2-3: (expert, token)
 *             pairs sorted by expert, sum in selection order).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless marked (host).  The caller allocates
 *     and owns every buffer; the library keeps no pointer after a call returns
 *     and never allocates, frees or synchronises.  Every call only enqueues
 *     kernels on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *     default stream).
 *   - Arguments are validated on the host before any launch; on a bad
 *     argument the call returns RL_ERR_INVALID (or RL_ERR_UNSUPPORTED for a
 *     shape outside the supported set) and launches nothing.  RL_ERR_CUDA
 *     reports a launch failure.  rl_last_error() gives a message for the last
 *     non-OK status of the calling thread.  Nothing aborts or prints.
 *   - `ctrl` is a 2-word int32 device control block owned by the caller:
 *       ctrl[0] = early-out layer, RL_NO_EARLY_OUT when no layer missed;
 *       ctrl[1] = device error bits (RL_DEVERR_*), 0 when healthy.
 *     The caller initialises it and reads it after synchronising.  rl_route at
 *     layer l returns at once on the device when ctrl[0] < l; every other call
 *     for layer l returns at once when ctrl[0] <= l.  Device-side problems
 *     (misaligned slot, bounded wait that ran out) set a bit in ctrl[1] and
 *     skip the affected work; they never trap.
 *   - Quantized format: a matrix is stored flat and row-major as consecutive
 *     66-byte blocks of 256 values: bytes 0-1 = fp16 scale d (little-endian),
 *     then 32 groups of (uint8 index into the 256 x 8 int8 codebook, uint8
 *     sign mask); value j of a group = d * codebook[idx][j] * (bit j of the
 *     sign mask ? -1 : +1).  An expert record is [gate I x H | up I x H |
 *     down H x I] back to back (rl_record_bytes), at a 16-byte aligned slot
 *     address.  Expert output o = down(silu(gate x) * (up x)).
 *   - Empty input: rl_rmsnorm, rl_route, rl_resolve_slots, rl_build_pairs and
 *     moe_prefill_chunk(_f32) accept T = 0.  Once the shape and the layer are
 *     valid they return RL_OK without reading their per-token buffers, which
 *     may then be NULL; offs and ctrl are still required where a call takes
 *     them, and rl_build_pairs still writes offs = 0.
 *   - Supported shapes: hidden in {256, 512, 1024, 2048}; inter in {128, 256,
 *     512, 1024, 2048}; 1 <= top_k <= 16; top_k <= n_experts <= 512;
 *     top_k * inter <= 16384; n_layers >= 1.
 */
#ifndef RL_MOE_H
#define RL_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rl_status {
    RL_OK = 0,
    RL_ERR_INVALID = 1,     /* bad argument; nothing launched */
    RL_ERR_UNSUPPORTED = 2, /* shape outside the supported set; nothing launched */
    RL_ERR_CUDA = 3,        /* a kernel launch failed */
    RL_ERR_TIMEOUT = 4      /* reserved for host-visible bounded-wait expiry */
} rl_status;

#define RL_NO_EARLY_OUT 0x7fffffff
#define RL_ABI_VERSION 1

/* device error bits in ctrl[1] */
#define RL_DEVERR_SLOT_ALIGN 1   /* a non-zero slot address was not 16-byte aligned */
#define RL_DEVERR_WAIT_TIMEOUT 2 /* a bounded on-chip wait ran out of iterations */
#define RL_DEVERR_BAD_ID 4       /* an expert id outside [0, n_experts) was read */
#define RL_DEVERR_MISSING 8      /* an expert kernel met a zero (absent) slot */
#define RL_DEVERR_RANGE 16       /* a fixed-point sum met a term outside its range: a router partial
                                    (moe_decode_stack) or a group of 8 squares of the RMSNorm
                                    (|x| beyond about 1400; rl_route, moe_decode, moe_decode_stack) */
#define RL_DEVERR_NAN 32         /* a router logit was NaN; NaN ranks below every number (never
                                    selected while K numbers remain), so inputs holding NaN
                                    are refused through this bit */

/* (host) model shape, passed by pointer to every call */
typedef struct rl_moe_shape {
    int32_t hidden;    /* H: token width */
    int32_t n_experts; /* E: routed experts per layer */
    int32_t top_k;     /* K: experts selected per token */
    int32_t inter;     /* I: expert intermediate width */
    int32_t n_layers;  /* L: layers covered by the residency table */
} rl_moe_shape;

int32_t rl_abi_version(void);
/* Message for the last non-OK status returned to the calling thread ("" if none). */
const char *rl_last_error(void);
/* Bytes of one expert record: 3 * hidden * inter / 256 * 66. 0 for an invalid shape. */
size_t rl_record_bytes(const rl_moe_shape *shp);

/*
 * rl_rmsnorm - unit-gain RMSNorm of T rows of width H:
 *   xn[t][h] = x[t][h] * r_t,  r_t = 1 / sqrt(mean_h(x[t][h]^2) + eps), computed in f32.
 * x, xn: [T][H] f32 row-major, 16-byte aligned (may alias).  H a multiple of 256; T >= 0.
 * mean(x^2) is summed exactly and in no particular order: the squares of each group of 8
 * consecutive values are added in a fixed f32 tree, each group sum is rounded to a multiple of
 * 2^-30 and the groups are added as 64-bit integers.  rl_route, moe_decode and
 * moe_decode_stack (which adds the groups of its CTAs' slices of x) compute the very same r_t
 * when they normalise their input on the fly (norm_eps >= 0).  A group sum of 2^25 or more
 * (|x| beyond about 1400) counts as 2^25; the calls with a control block then set
 * RL_DEVERR_RANGE.
 */
rl_status rl_rmsnorm(const float *x, float *xn, int32_t T, int32_t H, float eps, void *stream);

/*
 * rl_route - router for T tokens of one layer ("Red Lite dev21", "What changed": rl_route).
 *   xn = x (norm_eps < 0) or RMSNorm(x) with unit gain and that eps (norm_eps >= 0)
 *   logits[t][e] = sum_h w_router[e][h] * xn[t][h] (+ bias[e])          f32
 *   ids[t][0..K-1]: the K largest logits in descending order; equal values (-0.0 == +0.0)
 *                   go to the lower expert index
 *   weights[t][k] = exp(l_k - l_0) / sum_j exp(l_j - l_0) over the selection   f32
 *   slots[t][k]   = residency[layer][ids[t][k]]   (0 = not resident)
 *   miss[layer]  += number of (t, k) with slots[t][k] == 0   (atomic, exact)
 *   if that number > 0: ctrl[0] = min(ctrl[0], layer)
 *     ("Red Lite dev23", "What changed", item 1: the router raises the flag at layer f).
 * xn [T][H] f32; w_router [E][H] f32 row-major; bias [E] f32 or NULL; residency
 * [n_layers][E] uint64 slot addresses; ids int32 [T][K]; weights f32 [T][K]; slots uint64 [T][K];
 * miss uint32 [n_layers] (accumulated; the caller zeroes it); logits_out f32 [T][E] or NULL.
 * ws: scratch of rl_route_workspace_bytes(shp, T) bytes, 16-byte aligned; it must be
 * zero-filled before its first use (it holds a completion counter that every call leaves at
 * zero); calls that share a workspace must not overlap on the GPU.
 * x, w_router: 16-byte aligned.  0 <= layer < n_layers, T >= 0.
 */
size_t rl_route_workspace_bytes(const rl_moe_shape *shp, int32_t T);
rl_status rl_route(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *x, float norm_eps,
                   const float *w_router, const float *bias, const uint64_t *residency,
                   int32_t *ids, float *weights, uint64_t *slots, uint32_t *miss, int32_t *ctrl,
                   float *logits_out, void *ws, size_t ws_bytes, void *stream);

/*
 * rl_resolve_slots - slots[t][k] = residency[layer][ids[t][k]] for T tokens, with no miss
 * counting and no early-out check: re-resolves a layer's slots after its missing experts
 * were filled ("Red Lite dev23", "What changed", item 1: layer f's misses are loaded and
 * run with the ids the GPU selected).  ids int32 [T][K], slots uint64 [T][K].
 */
rl_status rl_resolve_slots(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids,
                           const uint64_t *residency, uint64_t *slots, void *stream);

/*
 * rl_fill_missing - the fill of layer `layer`'s absent selected experts, done by the device
 * ("Red Lite dev23", "What changed", item 1: the layer's missing experts are loaded and the
 * layer runs with the experts the router picked), with no host round trip:
 *   for each distinct expert e with some selection (t, k) of the layer whose slot is 0:
 *     copy the record (rl_record_bytes) from src[layer][e] to dst[layer][e],
 *     residency[layer][e] = dst[layer][e], *filled += 1;
 *   if any: *first_early_out = min(*first_early_out, layer) and, if ctrl[0] == layer,
 *     ctrl[0] = RL_NO_EARLY_OUT (the layer's experts then run);
 *   then slots[t][k] = residency[layer][ids[t][k]] for every selection.
 * Call after rl_route(layer) on the same stream; miss[layer] keeps rl_route's count.
 * ids int32 [T][K]; slots uint64 [T][K] (in/out); residency uint64 [n_layers][E] (in/out);
 * src, dst uint64 [n_layers][E]: record addresses the device can read (src: e.g. page-locked
 * host memory through rl_host_device_pointer) and HBM slots, 16-byte aligned, 0 where there is
 * none (a needed expert without one sets RL_DEVERR_MISSING, a misaligned one
 * RL_DEVERR_SLOT_ALIGN; it stays absent); filled uint32 [1] and first_early_out int32 [1]
 * accumulate.  ws: rl_fill_workspace_bytes(shp) bytes, 16-byte aligned, zero-filled before its
 * first use (every call leaves it so).
 */
size_t rl_fill_workspace_bytes(const rl_moe_shape *shp);
rl_status rl_fill_missing(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids, uint64_t *slots,
                          uint64_t *residency, const uint64_t *src, const uint64_t *dst, uint32_t *filled,
                          int32_t *first_early_out, int32_t *ctrl, void *ws, size_t ws_bytes, void *stream);

/*
 * rl_host_device_pointer - (host) the device address of page-locked host memory (host pointer
 * `host`), for rl_fill_missing's src.  RL_ERR_INVALID when `host` is not page-locked memory
 * the device can read.
 */
rl_status rl_host_device_pointer(const void *host, uint64_t *device);

/*
 * moe_decode - routed experts of ONE token ("Red Lite dev21", "What changed": the
 * single-token expert kernels read the slot table and weights rl_route wrote):
 *   y[h] = (accumulate ? y[h] : 0) + sum_{k=0..K-1, in order} weights[k] * o_k[h],
 *   o_k = down_k(silu(gate_k xn) * (up_k xn)), expert k at slots[k],
 *   xn = x (norm_eps < 0) or RMSNorm(x) with unit gain and that eps (norm_eps >= 0).
 * f32 CUDA-core arithmetic.  x [H] f32 (16-byte aligned); slots uint64 [K]; weights f32 [K];
 * codebook int8 [256][8]; y [H] f32 (accumulate = 1 adds into y, e.g. the residual stream;
 * y may be x); skip when ctrl[0] <= layer.
 * A zero slot sets RL_DEVERR_MISSING and leaves y unchanged.
 * ws: scratch of moe_decode_workspace_bytes(shp) bytes (K * inter f32 for h).
 */
size_t moe_decode_workspace_bytes(const rl_moe_shape *shp);
rl_status moe_decode(const rl_moe_shape *shp, int32_t layer, const float *x, float norm_eps, const uint64_t *slots,
                     const float *weights, const int8_t *codebook, float *y, int32_t accumulate,
                     int32_t *ctrl, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_decode_static - moe_decode with no workspace argument, for callers that cannot
 * allocate device memory: for instance a plugin or extension hosted by another program that
 * owns every device allocation and only passes in the tensors of the call, or a serving loop
 * that forbids allocation after start-up.  The K * inter floats of h scratch that moe_decode
 * takes from `ws` come instead from a fixed array inside the library
 * (RL_STATIC_SCRATCH_FLOATS floats = 64 KB, held on every device that loads the library until
 * the process exits).  The arguments and results are those of moe_decode.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - Every call on a device shares the one array: calls that overlap on the GPU (other
 *     streams, other host threads) race; serialise them.
 *   - top_k * inter above RL_STATIC_SCRATCH_FLOATS returns RL_ERR_UNSUPPORTED (with the
 *     supported shapes it always fits).
 * The Red Lite pages have no counterpart of this entry point.
 */
#define RL_STATIC_SCRATCH_FLOATS 16384
rl_status moe_decode_static(const rl_moe_shape *shp, int32_t layer, const float *x, float norm_eps,
                            const uint64_t *slots, const float *weights, const int8_t *codebook, float *y,
                            int32_t accumulate, int32_t *ctrl, void *stream);

/*
 * moe_decode_stack - a run of layers [layer0, layer0 + n_layers) of ONE token in a single
 * launch: for each layer l, the work of rl_route(l) then moe_decode(l) on the residual stream
 *   xn = RMSNorm(x) (norm_eps >= 0; norm_eps < 0: xn = x),  route as rl_route,
 *   x <- x + sum_{k in order} weights[l][k] * down_k(silu(gate_k xn) * (up_k xn)).
 * "Red Lite dev38 - decode: expert down-projection lanes and concurrent encoders", "Finding":
 * serialization between the small per-layer kernels was the dominant waste; here the layers
 * meet at on-chip grid barriers instead of kernel boundaries.  "Red Lite dev21", "What
 * changed": no host round trip between router and experts.  "Red Lite dev23", "What changed",
 * item 1: at the first layer f that selects an absent expert, ids/weights/slots[f] and miss[f]
 * are written, ctrl[0] = min(ctrl[0], f), and the launch stops with x = x_f (the input of
 * layer f), so the caller can fill, rl_resolve_slots(f), moe_decode(f) and resume at f + 1.
 * The expert arithmetic, the RMSNorm scale and the selection are those of the per-layer chain
 * rl_route + moe_decode; the router logits are summed differently: every CTA adds the dots of
 * its slice of x into 64-bit fixed-point accumulators (exact, order-independent sums of f32
 * partials of |p| < 2^19, resolution 2^-36), and logit = rs * sum + bias.  A partial outside
 * that range sets RL_DEVERR_RANGE (and counts as 0).  Results do not depend on how the layers
 * are split between calls.
 * x [H] f32 in/out (16-byte aligned); w_router [n_layers][E][H] f32; bias [n_layers][E] f32 or
 * NULL; residency [n_layers][E]; codebook int8 [256][8]; ids int32, weights f32, slots uint64:
 * [n_layers][K] (rows of the run are written); miss uint32 [n_layers] (accumulated);
 * logits_out f32 [n_layers][E] or NULL; x_hist f32 [n_layers][H] or NULL (x_l, the input of
 * each layer run, for validation).  Does nothing when ctrl[0] < layer0.
 * pregate (0 <= pregate <= min(32, E)): pre-gated expert prefetch ("Red Lite dev23 - per-layer
 * early-out and pre-gated expert prefetch", "What changed"): during layer l the next layer's
 * router is applied to layer l's normalised input, and the records of its `pregate` highest-
 * scoring resident experts are prefetched from HBM into L2, so that layer l + 1's expert copies
 * hit L2 when the prediction is right.  0 turns it off.  It never changes a result.
 * pregate_hits uint32 [n_layers] or NULL: for every layer after the first of the run, how
 * many of its K selected experts were in the previous layer's prediction.
 * ws: moe_decode_stack_workspace_bytes(shp) bytes, 16-byte aligned, zero-filled before its
 * first use; it holds a grid-barrier counter that grows across calls, so calls sharing one
 * workspace must not overlap on the GPU, and after a call that raised RL_DEVERR_WAIT_TIMEOUT
 * it must be zero-filled again.  One CTA runs on every SM (cooperative launch); a shape whose
 * CTA does not fit an SM returns RL_ERR_UNSUPPORTED before any launch.  Every on-chip wait is
 * bounded: on expiry RL_DEVERR_WAIT_TIMEOUT is set in ctrl[1] and the launch ends.
 * Bytes 64..71 of ws are test knobs and stay zero in normal use: the uint32 at byte 64, when
 * nonzero, replaces the poll limit of every wait of the launch; the int32 at byte 68, n > 0,
 * makes CTA n-1 leave before its first grid-barrier arrival, and n < 0 makes CTA -n-1 expect
 * 16 bytes more than its first router-column copy brings, so that the other CTAs' waits run
 * out (RL_DEVERR_WAIT_TIMEOUT) without any fault; zero-fill ws again afterwards.
 * Host side: the router's tensor-copy descriptor (built from the w_router address and the
 * shape, never from its contents) and the occupancy check are computed once per device and
 * kept, so repeated calls do no more host work than the launch; the launch may be captured in
 * a CUDA graph.
 */
size_t moe_decode_stack_workspace_bytes(const rl_moe_shape *shp);
rl_status moe_decode_stack(const rl_moe_shape *shp, int32_t layer0, int32_t n_layers, float *x, float norm_eps,
                           const float *w_router, const float *bias, const uint64_t *residency,
                           const int8_t *codebook, int32_t *ids, float *weights, uint64_t *slots,
                           uint32_t *miss, int32_t *ctrl, float *logits_out, float *x_hist, int32_t pregate,
                           uint32_t *pregate_hits, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_decode_layer - rl_route (T = 1) then moe_decode (accumulate = 0) of ONE token in ONE
 * launch, without a residual: y = sum_{k in order} weights[layer][k] * down_k(silu(gate_k xn)
 * * (up_k xn)) with xn = x (norm_eps < 0) or RMSNorm(x) (norm_eps >= 0).  It is the fused
 * kernel of moe_decode_stack run for a single layer, with y written instead of the residual
 * stream ("Red Lite dev21 - GPU-routed decode", "What changed": the router and the experts of
 * a decode token with no host round trip between them).  The router logits are summed across
 * CTAs in fixed point as in moe_decode_stack (they may differ from rl_route's in the last
 * bits).  If the layer selects an absent expert, ids/weights/slots[layer] and miss[layer] are
 * written, ctrl[0] = min(ctrl[0], layer) and y is not written, so the caller can fill,
 * rl_resolve_slots and moe_decode.  Does nothing when ctrl[0] < layer.
 * x [H] f32 (read only, 16-byte aligned); y [H] f32; the other arguments and ws as for
 * moe_decode_stack (ws: moe_decode_stack_workspace_bytes, zero-filled before its first use).
 */
rl_status moe_decode_layer(const rl_moe_shape *shp, int32_t layer, const float *x, float norm_eps,
                           const float *w_router, const float *bias, const uint64_t *residency,
                           const int8_t *codebook, int32_t *ids, float *weights, uint64_t *slots, uint32_t *miss,
                           int32_t *ctrl, float *logits_out, float *y, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_decode_stack_fill - moe_decode_stack (no pre-gating) where a layer that selects absent
 * experts does not stop the launch: the device fills them ("Red Lite dev23", "What changed",
 * item 1: the layer's missing experts are loaded and it runs with the experts the router
 * picked).  Every CTA copies its share of each missing record from fill_src[l][e] (an address
 * the device can read, e.g. page-locked host memory through rl_host_device_pointer) to
 * fill_dst[l][e] (its HBM slot); after a grid barrier residency[l][e] = slots[l][k] =
 * fill_dst[l][e], *filled += 1, and the layer runs.  miss[l] still counts the layer's misses;
 * ctrl[0] is not raised.  A missing expert without a source (0) or with a misaligned address
 * falls back to moe_decode_stack's stop.  fill_src, fill_dst uint64 [n_layers][E]; filled
 * uint32 [1] (accumulated).  Same results as the stop / fill / resume flow.
 */
rl_status moe_decode_stack_fill(const rl_moe_shape *shp, int32_t layer0, int32_t n_layers, float *x, float norm_eps,
                                const float *w_router, const float *bias, uint64_t *residency,
                                const int8_t *codebook, int32_t *ids, float *weights, uint64_t *slots,
                                uint32_t *miss, int32_t *ctrl, float *logits_out, float *x_hist,
                                const uint64_t *fill_src, const uint64_t *fill_dst, uint32_t *filled, void *ws,
                                size_t ws_bytes, void *stream);

/*
 * rl_build_pairs - (expert, token) pairs sorted by expert, stable in (t, k) order
 * ("Red Lite dev20", "What changed", item 3):
 *   offs[e] .. offs[e+1]-1 index the pairs of expert e; pair p is (pair_tok[p], pair_k[p]).
 * ids int32 [T][K]; offs uint32 [E+1]; pair_tok uint32 [T*K]; pair_k uint8 [T*K].
 * Skip when ctrl[0] <= layer.  ws: rl_build_pairs_workspace_bytes(shp, T) bytes (0 today).
 */
size_t rl_build_pairs_workspace_bytes(const rl_moe_shape *shp, int32_t T);
rl_status rl_build_pairs(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids,
                         uint32_t *offs, uint32_t *pair_tok, uint8_t *pair_k, int32_t *ctrl,
                         void *ws, size_t ws_bytes, void *stream);

/*
 * moe_prefill_chunk - routed experts of a chunk of T tokens over the expert-sorted pairs
 * ("Red Lite dev20", "What changed", item 3: batched gate/up and down over the pairs, then
 * each token's top-k accumulated in router selection order):
 *   y[t][h] = (accumulate ? y[t][h] : 0) + sum_{k in order} weights[t][k] * o_{t,k}[h].
 * Gate/up and down run as grouped GEMMs on the 5th-generation tensor cores (tcgen05,
 * accumulators in tensor memory) with 16-bit operands and f32 accumulation: the weights are
 * decoded to IEEE half precision (d * codebook value * sign, rounded once) straight into tensor
 * memory, the activations x and h are rounded to half precision (|x|, |h| must stay below
 * 65504).  Half precision keeps 11 significant bits against bfloat16's 8: with both operands
 * rounded, bfloat16 left the chunk's relative error near 3e-3 of a 5e-3 budget.
 * xn [T][H] f32; offs/pair_tok/pair_k from rl_build_pairs; slots uint64 [T][K] and weights
 * f32 [T][K] from rl_route; codebook int8 [256][8]; y [T][H] f32.  Skip when
 * ctrl[0] <= layer.  ws: moe_prefill_workspace_bytes(shp, T) bytes.
 * Limit of this build: with inter = 2048 the down GEMM's shared-memory layout (six activation
 * stages and two 66 KB weight buffers) exceeds the 227 KB a CTA may hold, and the call returns
 * RL_ERR_CUDA from the attribute request before any launch.
 */
size_t moe_prefill_workspace_bytes(const rl_moe_shape *shp, int32_t T);
rl_status moe_prefill_chunk(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn,
                            const uint32_t *offs, const uint32_t *pair_tok, const uint8_t *pair_k,
                            const uint64_t *slots, const float *weights, const int8_t *codebook,
                            float *y, int32_t accumulate, int32_t *ctrl, void *ws, size_t ws_bytes,
                            void *stream);

/*
 * moe_prefill_chunk_f32 - the same computation as moe_prefill_chunk with f32 CUDA-core
 * arithmetic throughout (a cross-check of the grouped path at f32 accuracy).  Same
 * arguments; ws: moe_prefill_workspace_bytes(shp, T) bytes.
 */
rl_status moe_prefill_chunk_f32(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn,
                                const uint32_t *offs, const uint32_t *pair_tok, const uint8_t *pair_k,
                                const uint64_t *slots, const float *weights, const int8_t *codebook,
                                float *y, int32_t accumulate, int32_t *ctrl, void *ws,
                                size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* RL_MOE_H */
