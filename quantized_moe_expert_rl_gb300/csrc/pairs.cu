// pairs.cu - (expert, token) pairs sorted by expert, stable in (token, k) order.
//
// Red Lite dev20 - batched prompt ingestion, "What changed" item 3: the chunk's routed
// experts run over (expert, token) pairs sorted by expert.  Here: one CTA of 32 warps does
// a counting sort.  Each warp owns a contiguous segment of the flat selections
// p = t*K + k; (1) per-warp histograms, (2) exclusive scan over experts -> offs, and a
// per-warp start cursor inside each expert's range, (3) each warp scatters its segment in
// order, 32 selections at a time, ranking equal experts inside the batch with match.any.
#include "rl_common.cuh"

namespace rl {

constexpr int kPairWarps = 32;

__global__ void __launch_bounds__(kPairWarps * 32) build_pairs_kernel(const int32_t *__restrict__ ids, int P, int K,
                                                                      int E, uint32_t *__restrict__ offs,
                                                                      uint32_t *__restrict__ pair_tok,
                                                                      uint8_t *__restrict__ pair_k, int32_t *ctrl,
                                                                      int layer) {
    extern __shared__ __align__(16) uint32_t hist[];  // [kPairWarps][E], then cursors in place
    __shared__ uint32_t scan_s[kPairWarps];
    if (ld_ctrl(ctrl) <= layer) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kPairWarps * E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int seg = (P + kPairWarps - 1) / kPairWarps;
    const int p_lo = min(P, warp * seg), p_hi = min(P, p_lo + seg);
    bool bad = false;
    for (int p = p_lo + lane; p < p_hi; p += 32) {
        int e = ids[p];
        if (e < 0 || e >= E) { bad = true; e = 0; }
        atomicAdd(&hist[warp * E + e], 1u);
    }
    if (__any_sync(kFull, bad) && lane == 0) dev_error(ctrl, RL_DEVERR_BAD_ID);
    __syncthreads();
    // exclusive scan of the per-expert totals (E <= 512 < blockDim) and per-warp cursors
    uint32_t tot = 0;
    if ((int)threadIdx.x < E)
        for (int w = 0; w < kPairWarps; ++w) tot += hist[w * E + threadIdx.x];
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scan_s[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = scan_s[lane], s = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += u;
        }
        scan_s[lane] = s - v;  // exclusive prefix of the warp totals
    }
    __syncthreads();
    if ((int)threadIdx.x < E) {
        const uint32_t start = scan_s[warp] + incl - tot;  // exclusive prefix over experts
        offs[threadIdx.x] = start;
        uint32_t c = start;
        for (int w = 0; w < kPairWarps; ++w) {
            const uint32_t n = hist[w * E + threadIdx.x];
            hist[w * E + threadIdx.x] = c;
            c += n;
        }
    }
    if (threadIdx.x == 0) offs[E] = (uint32_t)P;
    __syncthreads();
    uint32_t *cur = hist + warp * E;
    const unsigned lt = (1u << lane) - 1u;
    for (int base = p_lo; base < p_hi; base += 32) {
        const int p = base + lane;
        const bool on = p < p_hi;
        int e = on ? ids[p] : -1;
        if (on && (e < 0 || e >= E)) e = 0;
        const unsigned peers = __match_any_sync(kFull, e);
        if (on) {
            const uint32_t pos = cur[e] + __popc(peers & lt);
            pair_tok[pos] = (uint32_t)(p / K);
            pair_k[pos] = (uint8_t)(p % K);
        }
        __syncwarp();
        if (on && (peers & lt) == 0) cur[e] += __popc(peers);
        __syncwarp();
    }
}

}  // namespace rl

using namespace rl;

extern "C" size_t rl_build_pairs_workspace_bytes(const rl_moe_shape *shp, int32_t T) {
    (void)shp;
    (void)T;
    return 0;
}

extern "C" rl_status rl_build_pairs(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids,
                                    uint32_t *offs, uint32_t *pair_tok, uint8_t *pair_k, int32_t *ctrl, void *ws,
                                    size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers) return fail(RL_ERR_INVALID, "rl_build_pairs: layer %d", layer);
    // offs and ctrl are always needed (T = 0 still writes offs = 0); the per-selection
    // buffers only when there are selections
    if (T < 0 || !offs || !ctrl || (T > 0 && (!ids || !pair_tok || !pair_k)))
        return fail(RL_ERR_INVALID, "rl_build_pairs: bad arguments");
    const long long P = (long long)T * shp->top_k;
    if (P > (1ll << 30)) return fail(RL_ERR_UNSUPPORTED, "rl_build_pairs: %lld pairs", P);
    const int E = shp->n_experts;
    const size_t sm = (size_t)kPairWarps * E * sizeof(uint32_t);
    st = allow_smem((const void *)build_pairs_kernel, sm);
    if (st != RL_OK) return st;
    build_pairs_kernel<<<1, kPairWarps * 32, sm, as_stream(stream)>>>(ids, (int)P, shp->top_k, E, offs, pair_tok,
                                                                    pair_k, ctrl, layer);
    return check_launch("rl_build_pairs");
}
