// stack.cu - the ABI entry points of the fused decode kernel (moe_decode_stack,
// moe_decode_stack_fill, moe_decode_layer); the kernel itself is in stack_kernel.cuh, its
// device-fill variants are instantiated in stack_fill.cu.
#include "stack_kernel.cuh"

using namespace rl;

extern "C" size_t moe_decode_stack_workspace_bytes(const rl_moe_shape *shp) {
    if (!shp || shp->n_experts <= 0 || shp->top_k <= 0 || shp->inter <= 0) return 0;
    return 256 + 2 * align_up(2 * (size_t)shp->n_experts * sizeof(long long), 256) +
           align_up((size_t)shp->top_k * shp->inter * sizeof(float), 256);
}

static rl_status stack_entry(const rl_moe_shape *shp, int32_t layer0, int32_t n_layers, float *x, float norm_eps,
                             const float *w_router, const float *bias, uint64_t *residency, const int8_t *codebook,
                             int32_t *ids, float *weights, uint64_t *slots, uint32_t *miss, int32_t *ctrl,
                             float *logits_out, float *x_hist, int32_t pregate, uint32_t *pregate_hits,
                             const uint64_t *fill_src, const uint64_t *fill_dst, uint32_t *filled, float *y,
                             void *ws, size_t ws_bytes, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer0 < 0 || n_layers < 0 || layer0 + n_layers > shp->n_layers)
        return fail(RL_ERR_INVALID, "moe_decode_stack: layers [%d, %d) outside [0, %d)", layer0, layer0 + n_layers,
                    shp->n_layers);
    if (!x || !w_router || !residency || !codebook || !ids || !weights || !slots || !miss || !ctrl)
        return fail(RL_ERR_INVALID, "moe_decode_stack: NULL buffer");
    if (!ws || ws_bytes < moe_decode_stack_workspace_bytes(shp))
        return fail(RL_ERR_INVALID, "moe_decode_stack: workspace of %zu B needed, %zu given",
                    moe_decode_stack_workspace_bytes(shp), ws_bytes);
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router) | reinterpret_cast<uintptr_t>(ws) |
         reinterpret_cast<uintptr_t>(x_hist)) & 15)
        return fail(RL_ERR_INVALID, "moe_decode_stack: x, w_router, x_hist and ws must be 16-byte aligned");
    if (pregate < 0 || pregate > kStPredMax || pregate > shp->n_experts)
        return fail(RL_ERR_INVALID, "moe_decode_stack: pregate %d outside [0, min(%d, n_experts)]", pregate, kStPredMax);
    if (n_layers == 0) return RL_OK;
    StackArgs a = {};
    a.x = x;
    a.eps = norm_eps;
    a.W = w_router;
    a.bias = bias;
    a.table = residency;
    a.codebook = codebook;
    a.ids = ids;
    a.weights = weights;
    a.slots = slots;
    a.miss = miss;
    a.ctrl = ctrl;
    a.logits_out = logits_out;
    a.x_hist = x_hist;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    a.ctr = reinterpret_cast<unsigned long long *>(w8);
    a.ss = reinterpret_cast<long long *>(w8 + 128);
    const size_t accb = align_up(2 * (size_t)shp->n_experts * sizeof(long long), 256);
    a.acc = reinterpret_cast<long long *>(w8 + 256);
    a.acc_pg = reinterpret_cast<long long *>(w8 + 256 + accb);
    a.h = reinterpret_cast<float *>(w8 + 256 + 2 * accb);
    a.pg_hits = pregate_hits;
    a.pregate = pregate;
    a.table_w = fill_src ? residency : nullptr;
    a.fill_src = fill_src;
    a.fill_dst = fill_dst;
    a.filled = filled;
    a.y = y;
    a.layer0 = layer0;
    a.nl = n_layers;
    a.n_layers = shp->n_layers;
    a.H = shp->hidden;
    a.E = shp->n_experts;
    a.K = shp->top_k;
    a.I = shp->inter;
    cudaStream_t s = as_stream(stream);
    return fill_src ? launch_stack_fill(a, s) : launch_stack_any<false>(a, s);
}

extern "C" rl_status moe_decode_stack(const rl_moe_shape *shp, int32_t layer0, int32_t n_layers, float *x,
                                      float norm_eps, const float *w_router, const float *bias,
                                      const uint64_t *residency, const int8_t *codebook, int32_t *ids,
                                      float *weights, uint64_t *slots, uint32_t *miss, int32_t *ctrl,
                                      float *logits_out, float *x_hist, int32_t pregate, uint32_t *pregate_hits,
                                      void *ws, size_t ws_bytes, void *stream) {
    // without fill tables the residency table is only read
    return stack_entry(shp, layer0, n_layers, x, norm_eps, w_router, bias, const_cast<uint64_t *>(residency),
                       codebook, ids, weights, slots, miss, ctrl, logits_out, x_hist, pregate, pregate_hits, nullptr,
                       nullptr, nullptr, nullptr, ws, ws_bytes, stream);
}

extern "C" rl_status moe_decode_stack_fill(const rl_moe_shape *shp, int32_t layer0, int32_t n_layers, float *x,
                                           float norm_eps, const float *w_router, const float *bias,
                                           uint64_t *residency, const int8_t *codebook, int32_t *ids, float *weights,
                                           uint64_t *slots, uint32_t *miss, int32_t *ctrl, float *logits_out,
                                           float *x_hist, const uint64_t *fill_src, const uint64_t *fill_dst,
                                           uint32_t *filled, void *ws, size_t ws_bytes, void *stream) {
    if (!fill_src || !fill_dst || !filled) return fail(RL_ERR_INVALID, "moe_decode_stack_fill: NULL fill argument");
    return stack_entry(shp, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids, weights, slots,
                       miss, ctrl, logits_out, x_hist, 0, nullptr, fill_src, fill_dst, filled, nullptr, ws, ws_bytes,
                       stream);
}

extern "C" rl_status moe_decode_layer(const rl_moe_shape *shp, int32_t layer, const float *x, float norm_eps,
                                      const float *w_router, const float *bias, const uint64_t *residency,
                                      const int8_t *codebook, int32_t *ids, float *weights, uint64_t *slots,
                                      uint32_t *miss, int32_t *ctrl, float *logits_out, float *y, void *ws,
                                      size_t ws_bytes, void *stream) {
    if (!y) return fail(RL_ERR_INVALID, "moe_decode_layer: NULL y");
    // x is only read in this mode (the kernel writes y instead of the residual stream)
    return stack_entry(shp, layer, 1, const_cast<float *>(x), norm_eps, w_router, bias,
                       const_cast<uint64_t *>(residency), codebook, ids, weights, slots, miss, ctrl, logits_out,
                       nullptr, 0, nullptr, nullptr, nullptr, nullptr, y, ws, ws_bytes, stream);
}
