// prefill_common.cu - shared checks, workspace size and the ordered per-token combine.
//
// Red Lite dev20 - batched prompt ingestion, "What changed" item 3: each token's top-k
// outputs are accumulated in router selection order (the same order as decode).
#include "prefill_common.cuh"

namespace rl {

rl_status prefill_check(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn, const uint32_t *offs,
                        const uint32_t *pair_tok, const uint8_t *pair_k, const uint64_t *slots,
                        const float *weights, const int8_t *codebook, float *y, int32_t accumulate,
                        int32_t *ctrl, void *ws, size_t ws_bytes, const char *who, PrefillArgs *a) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers) return fail(RL_ERR_INVALID, "%s: layer %d outside [0,%d)", who, layer, shp->n_layers);
    if (T < 0) return fail(RL_ERR_INVALID, "%s: T=%d", who, T);
    if (!offs || !ctrl || (T > 0 && (!xn || !pair_tok || !pair_k || !slots || !weights || !codebook || !y)))
        return fail(RL_ERR_INVALID, "%s: NULL required buffer", who);
    if ((long long)T * shp->top_k > (1ll << 30)) return fail(RL_ERR_UNSUPPORTED, "%s: too many pairs", who);
    PrefillWs L(T, shp->hidden, shp->top_k, shp->inter, shp->n_experts);
    if (T > 0 && (!ws || ws_bytes < L.total))
        return fail(RL_ERR_INVALID, "%s: workspace of %zu B needed, %zu given", who, L.total, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(xn) | reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(y)) & 15)
        return fail(RL_ERR_INVALID, "%s: xn, y and ws must be 16-byte aligned", who);
    a->layer = layer; a->T = T; a->H = shp->hidden; a->E = shp->n_experts; a->K = shp->top_k; a->I = shp->inter;
    a->P = T * shp->top_k; a->accumulate = accumulate;
    a->xn = xn; a->offs = offs; a->pair_tok = pair_tok; a->pair_k = pair_k; a->slots = slots; a->weights = weights;
    a->codebook = codebook; a->y = y; a->ctrl = ctrl;
    uint8_t *w = static_cast<uint8_t *>(ws);
    a->hbuf = reinterpret_cast<float *>(w);
    a->outbuf = reinterpret_cast<float *>(w + L.h);
    a->xb16 = reinterpret_cast<uint16_t *>(w + L.h + L.out);
    a->hb16 = reinterpret_cast<uint16_t *>(w + L.h + L.out + L.xb);
    a->units = w + L.h + L.out + L.xb + L.hb;
    return RL_OK;
}

// y[t][h] = (acc ? y[t][h] : 0) + sum_{k = 0..K-1 in order} w[t][k] * out[t*K + k][h]
__global__ void __launch_bounds__(256) ordered_sum_kernel(const float *__restrict__ outbuf,
                                                          const float *__restrict__ weights, float *__restrict__ y,
                                                          int H, int K, int accumulate, const int32_t *ctrl,
                                                          int layer) {
    if (ld_ctrl(ctrl) <= layer) return;
    const int t = blockIdx.x;
    const float *ob = outbuf + (size_t)t * K * H;
    const float *w = weights + (size_t)t * K;
    for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
            const float wk = w[k];
            const float4 o = *reinterpret_cast<const float4 *>(ob + (size_t)k * H + c);
            acc.x = acc.x + wk * o.x; acc.y = acc.y + wk * o.y; acc.z = acc.z + wk * o.z; acc.w = acc.w + wk * o.w;
        }
        float4 *yp = reinterpret_cast<float4 *>(y + (size_t)t * H + c);
        if (accumulate) {
            const float4 r = *yp;
            acc.x = r.x + acc.x; acc.y = r.y + acc.y; acc.z = r.z + acc.z; acc.w = r.w + acc.w;
        }
        *yp = acc;
    }
}

rl_status launch_ordered_sum(const PrefillArgs &a, cudaStream_t s) {
    ordered_sum_kernel<<<a.T, 256, 0, s>>>(a.outbuf, a.weights, a.y, a.H, a.K, a.accumulate, a.ctrl, a.layer);
    return check_launch("moe_prefill ordered sum");
}

}  // namespace rl

extern "C" size_t moe_prefill_workspace_bytes(const rl_moe_shape *shp, int32_t T) {
    if (!shp || T < 0 || shp->hidden <= 0 || shp->top_k <= 0 || shp->inter <= 0) return 0;
    return rl::PrefillWs(T, shp->hidden, shp->top_k, shp->inter, shp->n_experts).total;
}
