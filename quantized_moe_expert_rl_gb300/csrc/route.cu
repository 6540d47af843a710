// route.cu - RMSNorm, router logits (f32), top-k selection with renormalised weights,
// residency lookup, per-layer miss count and early-out flag.
//
// Red Lite dev21 - GPU-routed decode (full residency), "What changed": rl_route selects the
// top-k on the GPU by logit with ties to the lower index, renormalises the weights over the
// selection, looks each expert up in the layers x experts residency table and writes the slot
// table, the weights and a per-layer miss count.
// Red Lite dev23 - per-layer early-out, "What changed" item 1: the router raises the flag at
// the first layer that selects a non-resident expert; later kernels then return at once.
//
// One token (decode): one kernel.  Each CTA owns 4 router rows, which it moves into shared
// memory with one bulk copy BEFORE griddepcontrol.wait (the router weights depend on nothing
// the previous kernel writes), so the 4 MB of router weights stream in while the previous
// layer finishes.  After the wait each warp dots one row with xn held in registers; the last
// CTA to finish (completion counter) selects, looks up and writes the outputs.
// Many tokens (prefill): f32 tiled GEMM, then one warp per token selects.
#include "qdot.cuh"
#include "select.cuh"

namespace rl {

// ---------------------------------------------------------------------------------------------
// RMSNorm: one CTA per token; warp 0 computes the deterministic scale, all threads apply it.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *__restrict__ x, float *__restrict__ xn, int H,
                                                      float eps) {
    __shared__ float r_s;
    const float *xr = x + (size_t)blockIdx.x * H;
    if (threadIdx.x < 32) {
        const float r = rms_scale_warp(xr, H, eps);
        if (threadIdx.x == 0) r_s = r;
    }
    __syncthreads();
    const float r = r_s;
    float *yr = xn + (size_t)blockIdx.x * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) yr[i] = xr[i] * r;
}

// ---------------------------------------------------------------------------------------------
// One token: fused RMSNorm (optional) + logits + last-CTA selection.
// NV = H / 128 float4 columns per lane (lane l owns columns 4l + 128j, j < NV).
// ---------------------------------------------------------------------------------------------
constexpr int kR1Rows = 4;
constexpr int kR1Threads = 32 * kR1Rows;

template <int NV, bool NORM, int C>
__global__ void __launch_bounds__(kR1Threads) route1_kernel(const float *__restrict__ x, float eps,
                                                            const float *__restrict__ W,
                                                            const float *__restrict__ bias,
                                                            const uint64_t *__restrict__ table_row, int32_t *ids,
                                                            float *weights, uint64_t *slots, uint32_t *miss_l,
                                                            int32_t *ctrl, int layer, float *logits,
                                                            unsigned *counter, int E, int K) {
    constexpr int H = NV * 128;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    float *scale_s = reinterpret_cast<float *>(smem + 16);
    int *last_s = reinterpret_cast<int *>(smem + 20);
    float *Ws = reinterpret_cast<float *>(smem + 128);  // [kR1Rows][H]
    const int e0 = blockIdx.x * kR1Rows, nr = min(kR1Rows, E - e0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)(nr * H * sizeof(float));
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(Ws, W + (size_t)e0 * H, bytes, bar);
    }
    cta_sync();  // also rejoins warp 0 (its shuffles follow)
    pdl_wait();
    const bool skip = ld_ctrl(ctrl) < layer;
    float4 xv[NV];
    if (!skip) {
#pragma unroll
        for (int j = 0; j < NV; ++j) xv[j] = reinterpret_cast<const float4 *>(x)[lane + 32 * j];
        if (NORM && warp == 0) {
            bool range = false;
            const float r = rms_scale_warp(x, H, eps, &range);
            if (lane == 0) {
                *scale_s = r;
                if (range && blockIdx.x == 0) dev_error(ctrl, RL_DEVERR_RANGE);
            }
        }
    }
    cta_sync();
    // the router rows must have landed before the CTA may exit, whether it skips or not
    if (!mbar_wait_warp(bar, 0)) {
        if (threadIdx.x == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        return;
    }
    if (skip) return;
    pdl_trigger();
    if (warp < nr) {
        const float r = NORM ? *scale_s : 1.f;
        const float4 *wr = reinterpret_cast<const float4 *>(Ws + warp * H);
        unsigned long long a0 = 0, a1 = 0;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            float4 v = xv[j];
            if (NORM) { v.x *= r; v.y *= r; v.z *= r; v.w *= r; }
            const float4 w = wr[lane + 32 * j];
            a0 = ffma2(pack2(__float_as_uint(w.x), __float_as_uint(w.y)),
                       pack2(__float_as_uint(v.x), __float_as_uint(v.y)), a0);
            a1 = ffma2(pack2(__float_as_uint(w.z), __float_as_uint(w.w)),
                       pack2(__float_as_uint(v.z), __float_as_uint(v.w)), a1);
        }
        const float s = warp_sum(hsum2(a0) + hsum2(a1));
        if (lane == 0) logits[e0 + warp] = s + (bias ? bias[e0 + warp] : 0.f);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(counter, 1u);
        *last_s = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (!*last_s) return;
    __threadfence();
    __syncwarp();  // warp 0 rejoined after thread 0's arrival (warp_select is all shuffles and votes)
    if (warp == 0) {
        warp_select<C>(logits, table_row, ids, weights, slots, miss_l, ctrl, layer, E, K);
        if (lane == 0) *counter = 0u;  // every call leaves the counter at zero
    }
}

// ---------------------------------------------------------------------------------------------
// Many tokens, register-tiled: logits[t][e] = sum_h xn[t][h] W[e][h] with a 128 x 128 tile per
// CTA, 8 x 8 outputs per thread (rows ty*4 + {0..3} and 64 + ty*4 + {0..3}, columns likewise
// from tx), K in steps of 8 staged k-major in shared memory (double-buffered, the next step's
// global loads in flight during the current one).  Split-K over blockIdx.z when the tiles alone
// cannot fill the GPU: slice z writes its partial sums, and router_reduce_kernel adds the
// slices in order (then the bias).  Every output is one thread's sequential f32 FMA chain per
// slice, so the result is deterministic.
// ---------------------------------------------------------------------------------------------
constexpr int kSgT = 128, kSgBK = 8, kSgPad = 4;

__global__ void __launch_bounds__(256, 2) router_sgemm_kernel(const float *__restrict__ xn, const float *__restrict__ W,
                                                           const float *__restrict__ bias, float *__restrict__ out,
                                                           int T, int H, int E, int kslice, const int32_t *ctrl,
                                                           int layer) {
    if (ld_ctrl(ctrl) < layer) return;
    __shared__ __align__(16) float As[2][kSgBK][kSgT + kSgPad];
    __shared__ __align__(16) float Bs[2][kSgBK][kSgT + kSgPad];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int t0 = blockIdx.y * kSgT, e0 = blockIdx.x * kSgT;
    const int k_lo = blockIdx.z * kslice, k_hi = k_lo + kslice;
    // loader: thread -> (row tid / 2, 4 consecutive k at (tid % 2) * 4) of both tiles
    const int lr = tid >> 1, lk = (tid & 1) * 4;
    const bool a_ok = t0 + lr < T, b_ok = e0 + lr < E;
    const float *a_src = xn + (size_t)(a_ok ? t0 + lr : 0) * H + lk;
    const float *b_src = W + (size_t)(b_ok ? e0 + lr : 0) * H + lk;
    float4 av = make_float4(0.f, 0.f, 0.f, 0.f), bv = av;
    if (a_ok) av = *reinterpret_cast<const float4 *>(a_src + k_lo);
    if (b_ok) bv = *reinterpret_cast<const float4 *>(b_src + k_lo);
    auto stage = [&](int buf) {
        As[buf][lk + 0][lr] = av.x; As[buf][lk + 1][lr] = av.y; As[buf][lk + 2][lr] = av.z; As[buf][lk + 3][lr] = av.w;
        Bs[buf][lk + 0][lr] = bv.x; Bs[buf][lk + 1][lr] = bv.y; Bs[buf][lk + 2][lr] = bv.z; Bs[buf][lk + 3][lr] = bv.w;
    };
    stage(0);
    __syncthreads();
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    int buf = 0;
    for (int k0 = k_lo; k0 < k_hi; k0 += kSgBK) {
        const bool more = k0 + kSgBK < k_hi;
        if (more) {  // next step's loads in flight during this step's FMAs
            if (a_ok) av = *reinterpret_cast<const float4 *>(a_src + k0 + kSgBK);
            if (b_ok) bv = *reinterpret_cast<const float4 *>(b_src + k0 + kSgBK);
        }
#pragma unroll
        for (int kk = 0; kk < kSgBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
            stage(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }
    float *o = out + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
            if (e < E) o[(size_t)t * E + e] = gridDim.z == 1 ? acc[i][j] + (bias ? bias[e] : 0.f) : acc[i][j];
        }
    }
}

// logits = (slice 0 + slice 1 + ...) + bias, slices added in order
__global__ void __launch_bounds__(256) router_reduce_kernel(const float *__restrict__ part, const float *__restrict__ bias,
                                                            float *__restrict__ logits, int T, int E, int S,
                                                            const int32_t *ctrl, int layer) {
    if (ld_ctrl(ctrl) < layer) return;
    const size_t n = (size_t)T * E;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float v = part[i];
        for (int z = 1; z < S; ++z) v += part[(size_t)z * n + i];
        logits[i] = v + (bias ? bias[i % E] : 0.f);
    }
}

template <int C>
__global__ void __launch_bounds__(256) route_select_kernel(const float *__restrict__ logits,
                                                           const uint64_t *__restrict__ table_row, int32_t *ids,
                                                           float *weights, uint64_t *slots, uint32_t *miss_l,
                                                           int32_t *ctrl, int layer, int T, int E, int K) {
    if (ld_ctrl(ctrl) < layer) return;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const size_t o = (size_t)t * K;
    warp_select<C>(logits + (size_t)t * E, table_row, ids + o, weights + o, slots + o, miss_l, ctrl, layer, E, K);
}

__global__ void resolve_slots_kernel(const int32_t *__restrict__ ids, const uint64_t *__restrict__ table_row,
                                     uint64_t *__restrict__ slots, int n, int E) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int e = ids[i];
    slots[i] = (e >= 0 && e < E) ? table_row[e] : 0;
}

constexpr int kSgMaxSplit = 8, kSgMaxSms = 256;
// split-K factor of the many-token router GEMM: enough CTAs for two per SM (two fit: 119
// registers x 256 threads, 16.5 KB), K slices that stay multiples of the K step.  With one
// 8-warp CTA per SM the FMA pipes wait on the shared-memory loads.  The workspace is sized with
// kSgMaxSms, so it does not depend on the device it was sized on.
static int router_splits(int T, int E, int H, int sms) {
    if (T <= 1) return 1;
    const int tiles = ((T + kSgT - 1) / kSgT) * ((E + kSgT - 1) / kSgT);
    sms = std::min(sms, kSgMaxSms);
    int S = 1;
    while (S < kSgMaxSplit && tiles * S * 2 <= 2 * sms && H % (kSgBK * S * 2) == 0 && H / (S * 2) >= 64) S *= 2;
    return S;
}

struct RouteWs {  // [counter (256 B) | logits T*E | normalised input T*H (T > 1 with norm) | split-K partials]
    size_t logits, xn, part, total;
    RouteWs(int T, int E, int H, bool norm) {
        logits = 256;
        xn = logits + align_up((size_t)T * E * sizeof(float), 256);
        part = xn + (norm && T > 1 ? align_up((size_t)T * H * sizeof(float), 256) : 0);
        const int S = router_splits(T, E, H, kSgMaxSms);
        total = part + (S > 1 ? align_up((size_t)S * T * E * sizeof(float), 256) : 0);
    }
};

template <int NV, bool NORM>
static rl_status launch_route1(const float *x, float eps, const float *W, const float *bias, const uint64_t *row,
                               int32_t *ids, float *w, uint64_t *slots, uint32_t *miss_l, int32_t *ctrl, int layer,
                               float *logits, unsigned *counter, int E, int K, cudaStream_t s) {
    const size_t sm = 128 + (size_t)kR1Rows * NV * 128 * sizeof(float);
    const dim3 g((E + kR1Rows - 1) / kR1Rows), b(kR1Threads);
#define RL_R1(C)                                                                                                     \
    return launch_pdl(route1_kernel<NV, NORM, C>, g, b, sm, s, "rl_route", x, eps, W, bias, row, ids, w, slots,     \
                      miss_l, ctrl, layer, logits, counter, E, K)
    if (E <= 32) RL_R1(1);
    if (E <= 64) RL_R1(2);
    if (E <= 128) RL_R1(4);
    if (E <= 256) RL_R1(8);
    RL_R1(16);
#undef RL_R1
}

template <int NV>
static rl_status launch_route1_n(bool norm, const float *x, float eps, const float *W, const float *bias,
                                 const uint64_t *row, int32_t *ids, float *w, uint64_t *slots, uint32_t *miss_l,
                                 int32_t *ctrl, int layer, float *logits, unsigned *counter, int E, int K,
                                 cudaStream_t s) {
    if (norm)
        return launch_route1<NV, true>(x, eps, W, bias, row, ids, w, slots, miss_l, ctrl, layer, logits, counter, E,
                                       K, s);
    return launch_route1<NV, false>(x, eps, W, bias, row, ids, w, slots, miss_l, ctrl, layer, logits, counter, E, K,
                                    s);
}

}  // namespace rl

using namespace rl;

extern "C" rl_status rl_rmsnorm(const float *x, float *xn, int32_t T, int32_t H, float eps, void *stream) {
    if (T < 0 || H <= 0 || (H % 256)) return fail(RL_ERR_INVALID, "rl_rmsnorm: bad T=%d or H=%d (H a multiple of 256)", T, H);
    if (!(eps >= 0.f)) return fail(RL_ERR_INVALID, "rl_rmsnorm: eps must be >= 0");
    if (T == 0) return RL_OK;  // no rows: the buffers are not read (they may be NULL)
    if (!x || !xn) return fail(RL_ERR_INVALID, "rl_rmsnorm: NULL buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xn)) & 15)
        return fail(RL_ERR_INVALID, "rl_rmsnorm: buffers must be 16-byte aligned");
    rmsnorm_kernel<<<T, 256, 0, as_stream(stream)>>>(x, xn, H, eps);
    return check_launch("rl_rmsnorm");
}

extern "C" size_t rl_route_workspace_bytes(const rl_moe_shape *shp, int32_t T) {
    if (!shp || T < 0 || shp->n_experts <= 0 || shp->hidden <= 0) return 0;
    return RouteWs(T, shp->n_experts, shp->hidden, true).total;
}

extern "C" rl_status rl_route(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *x, float norm_eps,
                              const float *w_router, const float *bias, const uint64_t *residency, int32_t *ids,
                              float *weights, uint64_t *slots, uint32_t *miss, int32_t *ctrl, float *logits_out,
                              void *ws, size_t ws_bytes, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers)
        return fail(RL_ERR_INVALID, "rl_route: layer %d outside [0,%d)", layer, shp->n_layers);
    if (T < 0) return fail(RL_ERR_INVALID, "rl_route: T=%d", T);
    if (T == 0) return RL_OK;  // no tokens: nothing is read or written (buffers may be NULL)
    if ((long long)T * shp->top_k > (1ll << 30)) return fail(RL_ERR_UNSUPPORTED, "rl_route: too many selections");
    if (!x || !w_router || !residency || !ids || !weights || !slots || !miss || !ctrl)
        return fail(RL_ERR_INVALID, "rl_route: NULL required buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router) |
         reinterpret_cast<uintptr_t>(ws)) & 15)
        return fail(RL_ERR_INVALID, "rl_route: x, w_router and ws must be 16-byte aligned");
    const int H = shp->hidden, E = shp->n_experts, K = shp->top_k;
    const bool norm = norm_eps >= 0.f;
    const RouteWs L(T, E, H, norm);
    if (!ws || ws_bytes < L.total)
        return fail(RL_ERR_INVALID, "rl_route: workspace of %zu B needed, %zu given", L.total, ws_bytes);
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    unsigned *counter = reinterpret_cast<unsigned *>(w8);
    float *logits = logits_out ? logits_out : reinterpret_cast<float *>(w8 + L.logits);
    const uint64_t *row = residency + (size_t)layer * E;
    uint32_t *miss_l = miss + layer;
    cudaStream_t s = as_stream(stream);
    if (T == 1) {
        switch (H) {
            case 256: return launch_route1_n<2>(norm, x, norm_eps, w_router, bias, row, ids, weights, slots, miss_l,
                                                ctrl, layer, logits, counter, E, K, s);
            case 512: return launch_route1_n<4>(norm, x, norm_eps, w_router, bias, row, ids, weights, slots, miss_l,
                                                ctrl, layer, logits, counter, E, K, s);
            case 1024: return launch_route1_n<8>(norm, x, norm_eps, w_router, bias, row, ids, weights, slots, miss_l,
                                                 ctrl, layer, logits, counter, E, K, s);
            default: return launch_route1_n<16>(norm, x, norm_eps, w_router, bias, row, ids, weights, slots, miss_l,
                                                ctrl, layer, logits, counter, E, K, s);
        }
    }
    const float *src = x;
    if (norm) {
        float *xn = reinterpret_cast<float *>(w8 + L.xn);
        rmsnorm_kernel<<<T, 256, 0, s>>>(x, xn, H, norm_eps);
        src = xn;
    }
    {
        const int S = router_splits(T, E, H, sm_count());
        float *part = S > 1 ? reinterpret_cast<float *>(w8 + L.part) : logits;
        router_sgemm_kernel<<<dim3((E + kSgT - 1) / kSgT, (T + kSgT - 1) / kSgT, S), 256, 0, s>>>(
            src, w_router, bias, part, T, H, E, H / S, ctrl, layer);
        if (S > 1) {
            const size_t n = (size_t)T * E;
            router_reduce_kernel<<<(int)std::min<size_t>((n + 255) / 256, 2048), 256, 0, s>>>(part, bias, logits, T, E,
                                                                                            S, ctrl, layer);
        }
    }
    const dim3 g((T + 7) / 8), b(256);
    if (E <= 32) route_select_kernel<1><<<g, b, 0, s>>>(logits, row, ids, weights, slots, miss_l, ctrl, layer, T, E, K);
    else if (E <= 64) route_select_kernel<2><<<g, b, 0, s>>>(logits, row, ids, weights, slots, miss_l, ctrl, layer, T, E, K);
    else if (E <= 128) route_select_kernel<4><<<g, b, 0, s>>>(logits, row, ids, weights, slots, miss_l, ctrl, layer, T, E, K);
    else if (E <= 256) route_select_kernel<8><<<g, b, 0, s>>>(logits, row, ids, weights, slots, miss_l, ctrl, layer, T, E, K);
    else route_select_kernel<16><<<g, b, 0, s>>>(logits, row, ids, weights, slots, miss_l, ctrl, layer, T, E, K);
    return check_launch("rl_route");
}

extern "C" rl_status rl_resolve_slots(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids,
                                      const uint64_t *residency, uint64_t *slots, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers) return fail(RL_ERR_INVALID, "rl_resolve_slots: layer %d", layer);
    if (T < 0) return fail(RL_ERR_INVALID, "rl_resolve_slots: T=%d", T);
    if (T == 0) return RL_OK;  // no tokens: the buffers are not read (they may be NULL)
    if (!ids || !residency || !slots) return fail(RL_ERR_INVALID, "rl_resolve_slots: NULL buffer");
    if ((long long)T * shp->top_k > (1ll << 30)) return fail(RL_ERR_UNSUPPORTED, "rl_resolve_slots: too many selections");
    const int n = T * shp->top_k;
    resolve_slots_kernel<<<(n + 255) / 256, 256, 0, as_stream(stream)>>>(
        ids, residency + (size_t)layer * shp->n_experts, slots, n, shp->n_experts);
    return check_launch("rl_resolve_slots");
}
