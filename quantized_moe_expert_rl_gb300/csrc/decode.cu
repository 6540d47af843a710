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

#include "decode_rows.cuh"

namespace rl {

constexpr int kGuThreads = 1024;
constexpr int kDnRows = 16;

constexpr int kGuChunks = 4;  // row chunks per expert segment, each with its own mbarrier

struct GuLayout {
    int rowb, rmax;  // bytes of one H-wide row; max rows per CTA
    size_t tiles, part, total;
    __host__ __device__ GuLayout(int H, int I, int K, int G) {
        rowb = (int)matrix_bytes(1, H);
        const int U = gu_unit(H), units = K * I / U;
        rmax = ((units + G - 1) / G) * U;
        // gate and up rows of <= rmax pairs; >= 2 KB because it first stages the codebook
        tiles = std::max((size_t)2048, 2 * (size_t)rmax * rowb);
        part = align_up((size_t)rmax * 4 * sizeof(float), 16);  // [row][half][gate, up]
        total = 128 + kTabBytes + (size_t)H * sizeof(float) + part + tiles;
    }
};

// GPL = groups (8 values) per lane = H / (256 * SPLIT); SPLIT warps per (gate, up) row pair.
template <int GPL, int SPLIT, bool NORM>
__global__ void __launch_bounds__(kGuThreads) dec_gateup_kernel(const float *__restrict__ xin, float eps,
                                                                const uint64_t *__restrict__ slots,
                                                                const int8_t *__restrict__ codebook,
                                                                float *__restrict__ h, int32_t *ctrl, int layer,
                                                                int H, int I, int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [2 segments][kGuChunks]
    float *scale_s = reinterpret_cast<float *>(smem + 8 * 2 * kGuChunks);
    int *ok_s = reinterpret_cast<int *>(smem + 8 * 2 * kGuChunks + 4);
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 128);
    const GuLayout lay(H, I, K, gridDim.x);
    float *x_s = reinterpret_cast<float *>(smem + 128 + kTabBytes);
    float *part = x_s + H;
    // [seg 0 gate | seg 0 up | seg 1 gate | seg 1 up], n0 and n1 rows; every row count is a
    // multiple of gu_unit(H), so every sub-tile starts 16-byte aligned
    uint8_t *tiles = reinterpret_cast<uint8_t *>(part) + lay.part;
    const int U = gu_unit(H), units = K * I / U;
    const int p0 = (int)((long long)blockIdx.x * units / gridDim.x) * U;
    const int p1 = (int)((long long)(blockIdx.x + 1) * units / gridDim.x) * U;
    const int ka = p0 / I, kb = (p1 - 1) / I;  // at most two experts (p1 - p0 <= I)
    const int n0 = (ka == kb ? p1 : (ka + 1) * I) - p0, n1 = (p1 - p0) - n0;
    // chunk c of segment s holds rows [cut(s, c), cut(s, c + 1)) of the segment
    auto cut = [&](int seg, int c) { return ((seg == 0 ? n0 : n1) / U * c / kGuChunks) * U; };
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kGuChunks; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    build_pair_table(tab, codebook, nullptr);  // ends with __syncthreads
    pdl_wait();
    // independent loads first: the flag, the two slots, x
    const int flag = ld_ctrl(ctrl);
    uint64_t sa = 0, sb = 0;
    if (threadIdx.x < 32) {
        sa = __ldcg(slots + ka);
        sb = __ldcg(slots + kb);
    }
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(x_s)[i] = __ldcg(reinterpret_cast<const float4 *>(xin) + i);
    if (flag <= layer) return;
    if (threadIdx.x < 32) {
        const bool ok = sa != 0 && (sa & 15) == 0 && sb != 0 && (sb & 15) == 0;
        if (threadIdx.x == 0) {
            if (sa == 0 || (sa & 15)) dev_error(ctrl, sa == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
            if (sb == 0 || (sb & 15)) dev_error(ctrl, sb == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
            *ok_s = ok;
        }
        if (ok) {
            // lane i < 2 * kGuChunks issues chunk (seg = i / kGuChunks, c = i % kGuChunks):
            // its gate rows and its up rows, completion on bars[i]
            const int seg = threadIdx.x / kGuChunks, c = threadIdx.x % kGuChunks;
            if (threadIdx.x < 2 * kGuChunks) {
                const int n = seg == 0 ? n0 : n1;
                const int r0 = cut(seg, c), r1 = cut(seg, c + 1);
                if (r1 > r0) {
                    const size_t matb = matrix_bytes(I, H);
                    const uint8_t *base = reinterpret_cast<const uint8_t *>(seg == 0 ? sa : sb);
                    const int ia = seg == 0 ? p0 - ka * I : 0;  // first row of the segment in the expert
                    const uint32_t bytes = (uint32_t)((r1 - r0) * lay.rowb);
                    uint8_t *gdst = tiles + (seg == 0 ? 0 : 2 * (size_t)n0 * lay.rowb) + (size_t)r0 * lay.rowb;
                    mbar_arrive_expect_tx(&bars[threadIdx.x], 2 * bytes);
                    bulk_g2s(gdst, base + (size_t)(ia + r0) * lay.rowb, bytes, &bars[threadIdx.x]);
                    bulk_g2s(gdst + (size_t)n * lay.rowb, base + matb + (size_t)(ia + r0) * lay.rowb, bytes,
                             &bars[threadIdx.x]);
                }
            }
        }
    }
    cta_sync();  // x staged, ok_s written; warp 0 rejoined after its lane-dependent copy issue
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (NORM && warp == 0) {
        bool range = false;
        const float r = rms_scale_warp(x_s, H, eps, &range);
        if (lane == 0) {
            *scale_s = r;
            if (range && blockIdx.x == 0) dev_error(ctrl, RL_DEVERR_RANGE);
        }
    }
    cta_sync();
    if (!*ok_s) return;
    pdl_trigger();
    const int half = warp % SPLIT, team = warp / SPLIT;
    constexpr int kTeams = kGuThreads / 32 / SPLIT;
    // lane's 8*GPL consecutive inputs: columns half*H/SPLIT + lane*8*GPL ...
    const int c0 = half * (H / SPLIT) + lane * 8 * GPL;
    unsigned long long xv[4 * GPL];  // the lane's inputs as packed f32 pairs
    {
        const float r = NORM ? *scale_s : 1.f;
#pragma unroll
        for (int q = 0; q < 2 * GPL; ++q) {
            const float4 v = reinterpret_cast<const float4 *>(x_s + c0)[q];
            pack4(make_float4(v.x * r, v.y * r, v.z * r, v.w * r), &xv[2 * q]);
        }
    }
    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
    const int gl = c0 / 8, boff = (gl >> 5) * kBlockBytes, g0 = gl & 31;  // lane's groups inside the row
    unsigned ready = 0;  // bit i: bars[i] observed complete by this warp
    bool timed_out = false;
    auto locate = [&](int p, const uint8_t *&gb, const uint8_t *&ub) {
        const int seg = p - p0 < n0 ? 0 : 1;
        const int r = seg == 0 ? p - p0 : p - p0 - n0;
        const int n = seg == 0 ? n0 : n1;
        int c = 0;
        while (c + 1 < kGuChunks && r >= cut(seg, c + 1)) ++c;
        const int bi = seg * kGuChunks + c;
        if (!(ready & (1u << bi))) {
            if (!mbar_wait_warp(&bars[bi], 0)) timed_out = true;
            ready |= 1u << bi;
        }
        gb = tiles + (seg == 0 ? 0 : 2 * (size_t)n0 * lay.rowb) + (size_t)r * lay.rowb + boff;
        ub = gb + (size_t)n * lay.rowb;
    };
    for (int p = p0 + team; p < p1; p += 2 * kTeams) {
        const int q = p + kTeams;  // second row pair in flight
        const uint8_t *gb, *ub, *gb2 = nullptr, *ub2 = nullptr;
        locate(p, gb, ub);
        if (q < p1) locate(q, gb2, ub2);
        if (timed_out) break;
        float gv, uv, gv2 = 0.f, uv2 = 0.f;
        gu_row<GPL>(gb, ub, g0, xv, tabc, gv, uv);
        if (q < p1) gu_row<GPL>(gb2, ub2, g0, xv, tabc, gv2, uv2);
        gv = warp_sum(gv);
        uv = warp_sum(uv);
        gv2 = warp_sum(gv2);
        uv2 = warp_sum(uv2);
        if (lane == 0) {
            part[((p - p0) * 2 + half) * 2 + 0] = gv;
            part[((p - p0) * 2 + half) * 2 + 1] = uv;
            if (q < p1) {
                part[((q - p0) * 2 + half) * 2 + 0] = gv2;
                part[((q - p0) * 2 + half) * 2 + 1] = uv2;
            }
        }
        __syncwarp();  // rejoin before the next row's shuffles (see cta_sync)
    }
    if (timed_out && lane == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
    // Warm L2 with the down matrices the next kernel reads (CTA c takes the c-th slice of every
    // selected expert's down matrix); issued after this CTA's own rows are in shared memory.
    if (warp == 0 && lane < K && !timed_out) {
        const uint64_t sd = __ldcg(slots + lane);
        if (sd != 0 && (sd & 15) == 0) {
            const size_t matb = matrix_bytes(I, H);
            const size_t per = align_up((matb + gridDim.x - 1) / gridDim.x, 256);
            const size_t off = per * blockIdx.x;
            if (off < matb)
                prefetch_l2_bulk(reinterpret_cast<const uint8_t *>(sd) + 2 * matb + off,
                                 (uint32_t)std::min(per, matb - off));
        }
    }
    __syncthreads();
    if (timed_out) return;
    for (int t = threadIdx.x; t < p1 - p0; t += blockDim.x) h[p0 + t] = swiglu_part<SPLIT>(part + 4 * t);  // p = k*I + i
}

struct DnLayout {
    size_t tileb, total;
    __host__ __device__ DnLayout(int I, int K) {
        tileb = align_up(matrix_bytes(kDnRows, I), 16);
        // the tiles area first stages the 2 KB codebook
        total = 128 + kTabBytes + std::max((size_t)2048, K * tileb) + (size_t)K * kDnRows * sizeof(float);
    }
};

// Rows of I values: LPR lanes per row (min(32, I/8)), GPL groups per lane; two warps per
// expert, 8 rows each.
template <int GPL, int LPR>
__global__ void dec_down_kernel(const uint64_t *__restrict__ slots, const float *__restrict__ weights,
                                const int8_t *__restrict__ codebook, const float *__restrict__ h,
                                float *__restrict__ y, int accumulate, int32_t *ctrl, int layer, int H, int I,
                                int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 128);
    const DnLayout lay(I, K);
    uint8_t *tiles = smem + 128 + kTabBytes;
    float *o_s = reinterpret_cast<float *>(tiles + std::max((size_t)2048, K * lay.tileb));  // [K][kDnRows]
    const int r0 = blockIdx.x * kDnRows;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    build_pair_table(tab, codebook, nullptr);
    pdl_wait();
    // independent loads first: the flag, the K slots, this warp's slice of h
    const int flag = ld_ctrl(ctrl);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = warp >> 1, r_lo = (warp & 1) * (kDnRows / 2);  // two warps per expert
    const int sub = lane / LPR, sl = lane % LPR;
    constexpr int kRowsPerPass = 32 / LPR;
    uint64_t sk = 0;
    if (threadIdx.x < K) sk = __ldcg(slots + threadIdx.x);
    unsigned long long hv[4 * GPL];  // h of the warp's expert as packed f32 pairs
#pragma unroll
    for (int q = 0; q < 2 * GPL; ++q)
        pack4(__ldcg(reinterpret_cast<const float4 *>(h + (size_t)k * I + sl * 8 * GPL) + q), &hv[2 * q]);
    if (flag <= layer) return;
    const bool bad = threadIdx.x < K && (sk == 0 || (sk & 15));
    if (bad) dev_error(ctrl, sk == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
    if (__syncthreads_or(bad)) return;
    if (threadIdx.x < 32) {
        // kDnRows rows of I values start on a block boundary (kDnRows * I % 2048 == 0)
        const uint32_t bytes = (uint32_t)matrix_bytes(kDnRows, I);
        if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, bytes * K);
        __syncwarp();
        if (threadIdx.x < K) {
            const size_t off = 2 * matrix_bytes(I, H) + matrix_bytes(r0, I);
            bulk_g2s(tiles + threadIdx.x * lay.tileb, reinterpret_cast<const uint8_t *>(sk) + off, bytes, bar);
        }
    }
    pdl_trigger();
    if (!mbar_wait_warp(bar, 0)) {
        if (lane == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        return;
    }
    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
    const uint8_t *tile = tiles + k * lay.tileb;
#pragma unroll 2
    for (int rr = r_lo + sub; rr < r_lo + kDnRows / 2; rr += kRowsPerPass) {
        const float o = down_row<GPL, LPR>(tile, rr, I, sl, hv, tabc);
        if (sl == 0) o_s[k * kDnRows + rr] = o;
        __syncwarp();
    }
    __syncthreads();
    if (threadIdx.x < kDnRows) {
        const int r = r0 + threadIdx.x;
        const float acc = ordered_combine(weights, o_s + threadIdx.x, kDnRows, K);
        y[r] = (accumulate ? y[r] : 0.f) + acc;
    }
}

template <int GPL, int SPLIT>
static rl_status launch_gateup(const float *x, float eps, const uint64_t *slots, const int8_t *cb, float *h,
                               int32_t *ctrl, int layer, int H, int I, int K, cudaStream_t s) {
    const int U = gu_unit(H);
    const int G = std::min(sm_count(), K * I / U);
    const GuLayout lay(H, I, K, G);
    if ((size_t)U * lay.rowb % 16 != 0 || lay.total > 200 * 1024 || (K * I) % U != 0 || G < K)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode: gate/up tile geometry (H=%d, I=%d, K=%d)", H, I, K);
    if (eps >= 0.f)
        return launch_pdl(dec_gateup_kernel<GPL, SPLIT, true>, dim3(G), dim3(kGuThreads), lay.total, s,
                          "moe_decode gate/up", x, eps, slots, cb, h, ctrl, layer, H, I, K);
    return launch_pdl(dec_gateup_kernel<GPL, SPLIT, false>, dim3(G), dim3(kGuThreads), lay.total, s,
                      "moe_decode gate/up", x, eps, slots, cb, h, ctrl, layer, H, I, K);
}

template <int GPL, int LPR>
static rl_status launch_down(const uint64_t *slots, const float *w, const int8_t *cb, const float *h, float *y,
                             int acc, int32_t *ctrl, int layer, int H, int I, int K, cudaStream_t s) {
    const DnLayout lay(I, K);
    if (matrix_bytes(kDnRows, I) % 16 != 0 || (kDnRows * I) % 2048 != 0 || lay.total > 200 * 1024)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode: down tile geometry (I=%d, K=%d)", I, K);
    return launch_pdl(dec_down_kernel<GPL, LPR>, dim3(H / kDnRows), dim3(64 * K), lay.total, s, "moe_decode down",
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
        case 256: st = launch_gateup<1, 1>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        case 512: st = launch_gateup<2, 1>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        case 1024: st = launch_gateup<2, 2>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
        default: st = launch_gateup<4, 2>(xn, norm_eps, slots, codebook, h, ctrl, layer, H, I, K, s); break;
    }
    if (st != RL_OK) return st;
    switch (I) {  // I/8 groups per row
        case 128: return launch_down<1, 16>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        case 256: return launch_down<1, 32>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
        case 512: return launch_down<4, 16>(slots, weights, codebook, h, y, accumulate, ctrl, layer, H, I, K, s);
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
// every shape check_shape accepts fits the array, so the size check below only guards a
// future widening of the supported shapes
static_assert(RL_STATIC_SCRATCH_FLOATS >= rl::kMaxKxI, "the fixed h scratch must hold top_k * inter floats");

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
