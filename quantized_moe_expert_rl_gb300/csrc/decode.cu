// decode.cu - routed experts of one token: dequantizing GEMVs on the CUDA cores in f32.
//
// Red Lite dev21 - GPU-routed decode, "What changed": the single-token expert kernels read
// the slot table and weights that rl_route wrote, so no host round trip sits between the
// router and the experts.  Red Lite dev38 - decode lanes, "Changes" item 1 tunes the lane
// mapping of the same GEMVs on another GPU; here:
//
// Kernel 1 (gate/up): the K*I (expert, row) pairs are split evenly over one CTA per SM.  One
//   elected thread moves the CTA's rows of gate and of up into shared memory with bulk
//   asynchronous copies (completion on an mbarrier); each warp then takes whole rows, each
//   lane decodes 8*GPL consecutive values (see qdot.cuh) against xn held in registers:
//     h[k][i] = silu(gate_k[i] . xn) * (up_k[i] . xn)
// Kernel 2 (down + ordered combine): CTA = 16 rows of y, one warp per expert k with h_k in
//   registers; the K partial rows meet in shared memory and are summed in selection order:
//     y[r] = (acc ? y[r] : 0) + sum_{k in order} w_k * (down_k[r] . h_k)
// Both kernels are launched as programmatic dependents: the codebook table is built before
// griddepcontrol.wait (it depends on nothing the previous kernel writes), everything else
// after it.  With norm_eps >= 0 the input is the raw residual x and is RMS-normalised on the
// fly with the same deterministic scale rl_rmsnorm computes.
#include <algorithm>
#include <mutex>

#include "qdot.cuh"

namespace rl {

constexpr int kGuThreads = 512;
constexpr int kDnRows = 16;

// rows of the flat (expert, row) space handled together so that copies stay 16-byte multiples
__host__ __device__ inline int gu_unit(int H) { return H >= 2048 ? 1 : 2048 / H; }

struct GuLayout {
    int rowb, rmax;  // bytes of one H-wide row; max rows per CTA
    size_t total;
    __host__ __device__ GuLayout(int H, int I, int K, int G) {
        rowb = (int)matrix_bytes(1, H);
        const int U = gu_unit(H), units = K * I / U;
        rmax = ((units + G - 1) / G) * U;
        // gate and up rows of <= rmax pairs; >= 2 KB because it first stages the codebook
        total = 128 + kTabBytes + std::max((size_t)2048, 2 * (size_t)rmax * rowb);
    }
};

template <int GPL, bool NORM>
__global__ void __launch_bounds__(kGuThreads) dec_gateup_kernel(const float *__restrict__ xin, float eps,
                                                                const uint64_t *__restrict__ slots,
                                                                const int8_t *__restrict__ codebook,
                                                                float *__restrict__ h, int32_t *ctrl, int layer,
                                                                int H, int I, int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [2]
    float *scale_s = reinterpret_cast<float *>(smem + 16);
    int *ok_s = reinterpret_cast<int *>(smem + 20);
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 128);
    // [seg 0 gate | seg 0 up | seg 1 gate | seg 1 up], n0 and n1 rows; every row count is a
    // multiple of gu_unit(H), so every sub-tile starts 16-byte aligned
    uint8_t *tiles = smem + 128 + kTabBytes;
    const GuLayout lay(H, I, K, gridDim.x);
    const int U = gu_unit(H), units = K * I / U;
    const int p0 = (int)((long long)blockIdx.x * units / gridDim.x) * U;
    const int p1 = (int)((long long)(blockIdx.x + 1) * units / gridDim.x) * U;
    const int ka = p0 / I, kb = (p1 - 1) / I;  // at most two experts (p1 - p0 <= I)
    const int n0 = (ka == kb ? p1 : (ka + 1) * I) - p0, n1 = (p1 - p0) - n0;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    build_pair_table(tab, codebook, reinterpret_cast<uint2 *>(tiles));  // tiles are free until the copies
    pdl_wait();
    if (ld_ctrl(ctrl) <= layer) return;
    if (threadIdx.x == 0) {
        const uint64_t sa = slots[ka], sb = slots[kb];
        int ok = 1;
        if (sa == 0 || (sa & 15)) { dev_error(ctrl, sa == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN); ok = 0; }
        if (sb == 0 || (sb & 15)) { dev_error(ctrl, sb == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN); ok = 0; }
        *ok_s = ok;
        if (ok) {
            const size_t matb = matrix_bytes(I, H);
            const int ia = p0 - ka * I;
            const uint32_t b0 = (uint32_t)(n0 * lay.rowb);
            mbar_arrive_expect_tx(&bars[0], 2 * b0);
            const uint8_t *A = reinterpret_cast<const uint8_t *>(sa);
            bulk_g2s(tiles, A + (size_t)ia * lay.rowb, b0, &bars[0]);
            bulk_g2s(tiles + b0, A + matb + (size_t)ia * lay.rowb, b0, &bars[0]);
            if (n1 > 0) {
                const uint32_t b1 = (uint32_t)(n1 * lay.rowb);
                mbar_arrive_expect_tx(&bars[1], 2 * b1);
                const uint8_t *B = reinterpret_cast<const uint8_t *>(sb);
                bulk_g2s(tiles + 2 * b0, B, b1, &bars[1]);
                bulk_g2s(tiles + 2 * b0 + b1, B + matb, b1, &bars[1]);
            }
        }
    }
    // Warm L2 with the down matrices the next kernel reads: CTA c prefetches the c-th slice of
    // every selected expert's down matrix (slots are final once this kernel runs).
    if (threadIdx.x >= 32 && threadIdx.x < 32 + K) {
        const uint64_t sd = slots[threadIdx.x - 32];
        if (sd != 0 && (sd & 15) == 0) {
            const size_t matb = matrix_bytes(I, H);
            const size_t per = align_up((matb + gridDim.x - 1) / gridDim.x, 256);
            const size_t off = per * blockIdx.x;
            if (off < matb)
                prefetch_l2_bulk(reinterpret_cast<const uint8_t *>(sd) + 2 * matb + off,
                                 (uint32_t)std::min(per, matb - off));
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // lane's 8*GPL consecutive inputs as packed pairs
    unsigned long long xp[4 * GPL];
#pragma unroll
    for (int q = 0; q < 2 * GPL; ++q) {
        const float4 v = reinterpret_cast<const float4 *>(xin + lane * 8 * GPL)[q];
        xp[2 * q] = pack2(__float_as_uint(v.x), __float_as_uint(v.y));
        xp[2 * q + 1] = pack2(__float_as_uint(v.z), __float_as_uint(v.w));
    }
    if (NORM && warp == 0) {
        const float r = rms_scale_warp(xin, H, eps);
        if (lane == 0) *scale_s = r;
    }
    __syncthreads();
    if (!*ok_s) return;
    pdl_trigger();
    if (NORM) {
        const float r = *scale_s;
#pragma unroll
        for (int q = 0; q < 4 * GPL; ++q)
            xp[q] = pack2(__float_as_uint(__uint_as_float((uint32_t)xp[q]) * r),
                          __float_as_uint(__uint_as_float((uint32_t)(xp[q] >> 32)) * r));
    }
    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
    const int gl = lane * GPL, boff = (gl >> 5) * kBlockBytes, g0 = gl & 31;
    bool ready0 = false, ready1 = false;
    for (int p = p0 + warp; p < p1; p += kGuThreads / 32) {
        const int seg = p - p0 < n0 ? 0 : 1;
        bool &ready = seg == 0 ? ready0 : ready1;
        if (!ready) {
            if (!mbar_wait(&bars[seg], 0)) {
                if (lane == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
                return;
            }
            ready = true;
        }
        const int r = seg == 0 ? p - p0 : p - p0 - n0;
        const size_t nseg = seg == 0 ? n0 : n1;  // rows in this segment
        const uint8_t *gb = tiles + (seg == 0 ? 0 : 2 * (size_t)n0 * lay.rowb) + (size_t)r * lay.rowb + boff;
        const uint8_t *ub = gb + nseg * lay.rowb;
        unsigned long long ag0 = 0, ag1 = 0, au0 = 0, au1 = 0;
#pragma unroll
        for (int g = 0; g < GPL; g += 2) {
            ag0 = group_fma(*reinterpret_cast<const uint16_t *>(gb + 2 + 2 * (g0 + g)), &xp[4 * g], tabc, ag0);
            au0 = group_fma(*reinterpret_cast<const uint16_t *>(ub + 2 + 2 * (g0 + g)), &xp[4 * g], tabc, au0);
            if (g + 1 < GPL) {
                ag1 = group_fma(*reinterpret_cast<const uint16_t *>(gb + 4 + 2 * (g0 + g)), &xp[4 * (g + 1)], tabc,
                                ag1);
                au1 = group_fma(*reinterpret_cast<const uint16_t *>(ub + 4 + 2 * (g0 + g)), &xp[4 * (g + 1)], tabc,
                                au1);
            }
        }
        const float dg = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(gb));
        const float du = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(ub));
        const float gv = warp_sum(dg * (hsum2(ag0) + hsum2(ag1)));
        const float uv = warp_sum(du * (hsum2(au0) + hsum2(au1)));
        if (lane == 0) h[p] = silu(gv) * uv;  // p = k * I + i
    }
}

struct DnLayout {
    size_t tileb, total;
    __host__ __device__ DnLayout(int I, int K) {
        tileb = align_up(matrix_bytes(kDnRows, I), 16);
        // the tiles area first stages the 2 KB codebook
        total = 128 + kTabBytes + std::max((size_t)2048, K * tileb) + (size_t)K * kDnRows * sizeof(float);
    }
};

// Rows of I values: LPR lanes per row (min(32, I/8)), GPL groups per lane; one warp per expert.
template <int GPL, int LPR>
__global__ void dec_down_kernel(const uint64_t *__restrict__ slots, const float *__restrict__ weights,
                                const int8_t *__restrict__ codebook, const float *__restrict__ h,
                                float *__restrict__ y, int accumulate, int32_t *ctrl, int layer, int H, int I,
                                int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *ok_s = reinterpret_cast<int *>(smem + 16);
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 128);
    const DnLayout lay(I, K);
    uint8_t *tiles = smem + 128 + kTabBytes;
    float *o_s = reinterpret_cast<float *>(tiles + std::max((size_t)2048, K * lay.tileb));  // [K][kDnRows]
    const int r0 = blockIdx.x * kDnRows;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    build_pair_table(tab, codebook, reinterpret_cast<uint2 *>(tiles));  // tiles are free until the copies
    pdl_wait();
    if (ld_ctrl(ctrl) <= layer) return;
    if (threadIdx.x == 0) {
        int ok = 1;
        for (int k = 0; k < K; ++k) {
            const uint64_t s = slots[k];
            if (s == 0 || (s & 15)) { dev_error(ctrl, s == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN); ok = 0; }
        }
        *ok_s = ok;
        if (ok) {
            // kDnRows rows of I values start on a block boundary (kDnRows * I % 2048 == 0)
            const uint32_t bytes = (uint32_t)matrix_bytes(kDnRows, I);
            const size_t off = 2 * matrix_bytes(I, H) + matrix_bytes(r0, I);
            mbar_arrive_expect_tx(bar, bytes * K);
            for (int k = 0; k < K; ++k)
                bulk_g2s(tiles + k * lay.tileb, reinterpret_cast<const uint8_t *>(slots[k]) + off, bytes, bar);
        }
    }
    __syncthreads();
    if (!*ok_s) return;
    const int lane = threadIdx.x & 31, k = threadIdx.x >> 5;  // one warp per expert
    const int sub = lane / LPR, sl = lane % LPR;
    constexpr int kRowsPerPass = 32 / LPR;
    unsigned long long hp[4 * GPL];
#pragma unroll
    for (int q = 0; q < 2 * GPL; ++q) {
        const float4 v = reinterpret_cast<const float4 *>(h + (size_t)k * I + sl * 8 * GPL)[q];
        hp[2 * q] = pack2(__float_as_uint(v.x), __float_as_uint(v.y));
        hp[2 * q + 1] = pack2(__float_as_uint(v.z), __float_as_uint(v.w));
    }
    pdl_trigger();
    if (!mbar_wait(bar, 0)) {
        if (lane == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        return;
    }
    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
    const uint8_t *tile = tiles + k * lay.tileb;
#pragma unroll 2
    for (int rr = sub; rr < kDnRows; rr += kRowsPerPass) {
        const int gtile = rr * (I / 8) + sl * GPL;  // group index inside the tile
        const uint8_t *blk = tile + (gtile >> 5) * kBlockBytes;
        const int g0 = gtile & 31;
        unsigned long long a0 = 0, a1 = 0;
#pragma unroll
        for (int g = 0; g < GPL; g += 2) {
            a0 = group_fma(*reinterpret_cast<const uint16_t *>(blk + 2 + 2 * (g0 + g)), &hp[4 * g], tabc, a0);
            if (g + 1 < GPL)
                a1 = group_fma(*reinterpret_cast<const uint16_t *>(blk + 4 + 2 * (g0 + g)), &hp[4 * (g + 1)], tabc,
                               a1);
        }
        const float d = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        const float o = group_sum<LPR>(d * (hsum2(a0) + hsum2(a1)));
        if (sl == 0) o_s[k * kDnRows + rr] = o;
    }
    __syncthreads();
    if (threadIdx.x < kDnRows) {
        const int r = r0 + threadIdx.x;
        float acc = 0.f;
        for (int kk = 0; kk < K; ++kk) acc = acc + weights[kk] * o_s[kk * kDnRows + threadIdx.x];
        y[r] = (accumulate ? y[r] : 0.f) + acc;
    }
}

template <int GPL>
static rl_status launch_gateup(const float *x, float eps, const uint64_t *slots, const int8_t *cb, float *h,
                               int32_t *ctrl, int layer, int H, int I, int K, cudaStream_t s) {
    const int U = gu_unit(H);
    const int G = std::min(sm_count(), K * I / U);
    const GuLayout lay(H, I, K, G);
    if ((size_t)U * lay.rowb % 16 != 0 || lay.total > 200 * 1024 || (K * I) % U != 0)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode: gate/up tile geometry (H=%d, I=%d, K=%d)", H, I, K);
    if (eps >= 0.f)
        return launch_pdl(dec_gateup_kernel<GPL, true>, dim3(G), dim3(kGuThreads), lay.total, s,
                          "moe_decode gate/up", x, eps, slots, cb, h, ctrl, layer, H, I, K);
    return launch_pdl(dec_gateup_kernel<GPL, false>, dim3(G), dim3(kGuThreads), lay.total, s, "moe_decode gate/up",
                      x, eps, slots, cb, h, ctrl, layer, H, I, K);
}

template <int GPL, int LPR>
static rl_status launch_down(const uint64_t *slots, const float *w, const int8_t *cb, const float *h, float *y,
                             int acc, int32_t *ctrl, int layer, int H, int I, int K, cudaStream_t s) {
    const DnLayout lay(I, K);
    if (matrix_bytes(kDnRows, I) % 16 != 0 || (kDnRows * I) % 2048 != 0 || lay.total > 200 * 1024)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode: down tile geometry (I=%d, K=%d)", I, K);
    return launch_pdl(dec_down_kernel<GPL, LPR>, dim3(H / kDnRows), dim3(32 * K), lay.total, s, "moe_decode down",
                      slots, w, cb, h, y, acc, ctrl, layer, H, I, K);
}

}  // namespace rl

using namespace rl;

extern "C" size_t moe_decode_workspace_bytes(const rl_moe_shape *shp) {
    if (!shp || shp->top_k <= 0 || shp->inter <= 0) return 0;
    return align_up((size_t)shp->top_k * shp->inter * sizeof(float), 256);
}

extern "C" rl_status moe_decode(const rl_moe_shape *shp, int32_t layer, const float *xn, float norm_eps,
                                const uint64_t *slots, const float *weights, const int8_t *codebook, float *y,
                                int32_t accumulate, int32_t *ctrl, void *ws, size_t ws_bytes, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers)
        return fail(RL_ERR_INVALID, "moe_decode: layer %d outside [0,%d)", layer, shp->n_layers);
    if (!xn || !slots || !weights || !codebook || !y || !ctrl) return fail(RL_ERR_INVALID, "moe_decode: NULL buffer");
    if (!ws || ws_bytes < moe_decode_workspace_bytes(shp))
        return fail(RL_ERR_INVALID, "moe_decode: workspace of %zu B needed, %zu given",
                    moe_decode_workspace_bytes(shp), ws_bytes);
    if ((reinterpret_cast<uintptr_t>(xn) | reinterpret_cast<uintptr_t>(ws)) & 15)
        return fail(RL_ERR_INVALID, "moe_decode: xn and ws must be 16-byte aligned");
    const int H = shp->hidden, I = shp->inter, K = shp->top_k;
    float *h = static_cast<float *>(ws);
    cudaStream_t s = as_stream(stream);
    switch (H) {
        case 256: st = launch_gateup<1>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        case 512: st = launch_gateup<2>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        case 1024: st = launch_gateup<4>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        default: st = launch_gateup<8>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
    }
    if (st != RL_OK) return st;
    switch (I) {  // I/8 groups per row
        case 128: return launch_down<1, 16>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        case 256: return launch_down<1, 32>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        case 512: return launch_down<2, 32>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        case 1024: return launch_down<4, 32>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        default: return launch_down<8, 32>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
    }
}

// ---------------------------------------------------------------------------------------------
// moe_decode_static: moe_decode for callers that cannot hand the library any device memory
// of its own (see rl_moe.h).  The h scratch lives in this fixed device array instead of a
// caller workspace.  The array exists once per device that loads the library, for the life of
// the process; every call on a device shares it, so calls that overlap on the GPU race.  Each
// call overwrites every h entry it later reads, so nothing needs clearing between calls.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) float g_static_h[RL_STATIC_SCRATCH_FLOATS];

namespace rl {
// Device address of g_static_h on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is asked of the runtime once per device (with
// that device current) and cached.
static rl_status static_scratch(float **out) {
    static std::mutex mu;
    static float *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "moe_decode_static: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(RL_ERR_UNSUPPORTED, "moe_decode_static: device %d", dev);
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_h);
        if (e != cudaSuccess || !p)
            return fail(RL_ERR_CUDA, "moe_decode_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        addr[dev] = static_cast<float *>(p);
    }
    *out = addr[dev];
    return RL_OK;
}
}  // namespace rl

extern "C" rl_status moe_decode_static(const rl_moe_shape *shp, int32_t layer, const float *x, float norm_eps,
                                       const uint64_t *slots, const float *weights, const int8_t *codebook, float *y,
                                       int32_t accumulate, int32_t *ctrl, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if ((size_t)shp->top_k * shp->inter > RL_STATIC_SCRATCH_FLOATS)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode_static: top_k * inter = %d exceeds the fixed scratch of %d floats",
                    shp->top_k * shp->inter, RL_STATIC_SCRATCH_FLOATS);
    float *h = nullptr;
    st = static_scratch(&h);
    if (st != RL_OK) return st;
    return moe_decode(shp, layer, x, norm_eps, slots, weights, codebook, y, accumulate, ctrl, h,
                      (size_t)RL_STATIC_SCRATCH_FLOATS * sizeof(float), stream);
}
