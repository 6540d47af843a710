// prefill_f32.cu - routed experts of a chunk over the expert-sorted pairs, f32 CUDA cores.
//
// Red Lite dev20 - batched prompt ingestion, "What changed" item 3: batched gate/up and down
// over (expert, token) pairs sorted by expert, then each token's top-k accumulated in router
// selection order.  This f32 path is the accuracy cross-check of the tensor-core path; it
// shares its workspace layout and its ordered-sum kernel.
//
//   gate/up : CTA (expert e, 32 rows): h[p][i] = silu(gate_e[i] . xn[tok_p]) * (up_e[i] . xn[tok_p])
//   down    : CTA (expert e, 16 rows): out[t*K + k][r] = down_e[r] . h[p]      for pair p = (t, k)
//   combine : y[t] = (acc ? y[t] : 0) + sum_{k in order} w[t][k] * out[t*K + k]
#include "prefill_common.cuh"

namespace rl {

constexpr int kPfRows = 32;
constexpr int kPfDownRows = 16;
constexpr int kPfTok = 8;
constexpr int kPfThreads = 256;

__host__ __device__ static size_t gu_tile(int H) { return align_up((size_t)kPfRows * matrix_bytes(1, H), 16); }
__host__ __device__ static size_t gu_smem(int H) { return 16 + kGridBytes + 2 * gu_tile(H) + (size_t)kPfTok * H * sizeof(float); }
__host__ __device__ static size_t dn_tile(int I) { return align_up(matrix_bytes(kPfDownRows, I), 16); }
__host__ __device__ static size_t dn_smem(int I) { return 16 + kGridBytes + dn_tile(I) + (size_t)kPfTok * I * sizeof(float); }

template <int GPL>
__global__ void __launch_bounds__(kPfThreads) pf32_gateup_kernel(const float *__restrict__ xn,
                                                                 const uint32_t *__restrict__ offs,
                                                                 const uint32_t *__restrict__ pair_tok,
                                                                 const uint8_t *__restrict__ pair_k,
                                                                 const uint64_t *__restrict__ slots,
                                                                 const int8_t *__restrict__ codebook,
                                                                 float *__restrict__ hbuf, int32_t *ctrl, int layer,
                                                                 int H, int I, int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    if (ld_ctrl(ctrl) <= layer) return;
    const int e = blockIdx.x;
    const uint32_t p0 = offs[e], n = offs[e + 1] - p0;
    if (n == 0) return;
    const uint64_t slot = slots[(size_t)pair_tok[p0] * K + pair_k[p0]];
    if (slot == 0 || (slot & 15)) {
        if (threadIdx.x == 0) dev_error(ctrl, slot == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
        return;
    }
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int8_t *grid_s = reinterpret_cast<int8_t *>(smem + 16);
    uint8_t *gate_s = smem + 16 + kGridBytes;
    uint8_t *up_s = gate_s + gu_tile(H);
    float *x_s = reinterpret_cast<float *>(up_s + gu_tile(H));
    const size_t rowb = matrix_bytes(1, H), matb = matrix_bytes(I, H);
    const int i0 = blockIdx.y * kPfRows;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)(kPfRows * rowb);
        mbar_arrive_expect_tx(bar, 2 * bytes);
        const uint8_t *base = reinterpret_cast<const uint8_t *>(slot);
        bulk_g2s(gate_s, base + (size_t)i0 * rowb, bytes, bar);
        bulk_g2s(up_s, base + matb + (size_t)i0 * rowb, bytes, bar);
    }
    for (int i = threadIdx.x; i < kGridBytes / 8; i += blockDim.x)
        reinterpret_cast<uint2 *>(grid_s)[i] = reinterpret_cast<const uint2 *>(codebook)[i];
    __syncthreads();
    if (!mbar_wait_warp(bar, 0)) {
        if (threadIdx.x == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gl = lane * GPL, boff = (gl >> 5) * kBlockBytes, g0 = gl & 31;
    for (uint32_t j0 = 0; j0 < n; j0 += kPfTok) {
        const int nb = min((uint32_t)kPfTok, n - j0);
        __syncthreads();
        for (int i = threadIdx.x; i < nb * H / 4; i += blockDim.x) {
            const int jj = i / (H / 4), c = i % (H / 4);
            reinterpret_cast<float4 *>(x_s)[i] =
                reinterpret_cast<const float4 *>(xn + (size_t)pair_tok[p0 + j0 + jj] * H)[c];
        }
        __syncthreads();
        for (int r = warp; r < kPfRows; r += kPfThreads / 32) {
            const uint8_t *gb = gate_s + r * rowb + boff;
            const uint8_t *ub = up_s + r * rowb + boff;
            const float dg = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(gb));
            const float du = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(ub));
            for (int jj = 0; jj < nb; ++jj) {
                float xv[8 * GPL];
#pragma unroll
                for (int q = 0; q < 2 * GPL; ++q) {
                    const float4 v = reinterpret_cast<const float4 *>(x_s + (size_t)jj * H + lane * 8 * GPL)[q];
                    xv[4 * q] = v.x; xv[4 * q + 1] = v.y; xv[4 * q + 2] = v.z; xv[4 * q + 3] = v.w;
                }
                float g = warp_sum(dg * groups_dot<GPL>(gb, g0, xv, grid_s));
                float u = warp_sum(du * groups_dot<GPL>(ub, g0, xv, grid_s));
                if (lane == 0) hbuf[(size_t)(p0 + j0 + jj) * I + i0 + r] = silu(g) * u;
            }
        }
    }
}

template <int GPL, int LPR>
__global__ void __launch_bounds__(kPfThreads) pf32_down_kernel(const uint32_t *__restrict__ offs,
                                                               const uint32_t *__restrict__ pair_tok,
                                                               const uint8_t *__restrict__ pair_k,
                                                               const uint64_t *__restrict__ slots,
                                                               const int8_t *__restrict__ codebook,
                                                               const float *__restrict__ hbuf,
                                                               float *__restrict__ outbuf, int32_t *ctrl, int layer,
                                                               int H, int I, int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    if (ld_ctrl(ctrl) <= layer) return;
    const int e = blockIdx.x;
    const uint32_t p0 = offs[e], n = offs[e + 1] - p0;
    if (n == 0) return;
    const uint64_t slot = slots[(size_t)pair_tok[p0] * K + pair_k[p0]];
    if (slot == 0 || (slot & 15)) {
        if (threadIdx.x == 0) dev_error(ctrl, slot == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
        return;
    }
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int8_t *grid_s = reinterpret_cast<int8_t *>(smem + 16);
    uint8_t *tile = smem + 16 + kGridBytes;
    float *h_s = reinterpret_cast<float *>(tile + dn_tile(I));
    const size_t matb = matrix_bytes(I, H);
    const int r0 = blockIdx.y * kPfDownRows;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = (uint32_t)matrix_bytes(kPfDownRows, I);   // whole blocks (16*I % 2048 == 0)
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(tile, reinterpret_cast<const uint8_t *>(slot) + 2 * matb + matrix_bytes(r0, I), bytes, bar);
    }
    for (int i = threadIdx.x; i < kGridBytes / 8; i += blockDim.x)
        reinterpret_cast<uint2 *>(grid_s)[i] = reinterpret_cast<const uint2 *>(codebook)[i];
    __syncthreads();
    if (!mbar_wait_warp(bar, 0)) {
        if (threadIdx.x == 0) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kRowsPerPass = 32 / LPR;
    const int sub = lane / LPR, sl = lane % LPR;
    for (uint32_t j0 = 0; j0 < n; j0 += kPfTok) {
        const int nb = min((uint32_t)kPfTok, n - j0);
        __syncthreads();
        for (int i = threadIdx.x; i < nb * I / 4; i += blockDim.x)
            reinterpret_cast<float4 *>(h_s)[i] = reinterpret_cast<const float4 *>(hbuf + (size_t)(p0 + j0) * I)[i];
        __syncthreads();
        for (int rr = warp * kRowsPerPass + sub; rr < kPfDownRows; rr += (kPfThreads / 32) * kRowsPerPass) {
            const int gtile = rr * (I / 8) + sl * GPL;
            const uint8_t *blk = tile + (gtile >> 5) * kBlockBytes;
            const int g0 = gtile & 31;
            const float d = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
            for (int jj = 0; jj < nb; ++jj) {
                float hv[8 * GPL];
#pragma unroll
                for (int q = 0; q < 2 * GPL; ++q) {
                    const float4 v = reinterpret_cast<const float4 *>(h_s + (size_t)jj * I + sl * GPL * 8)[q];
                    hv[4 * q] = v.x; hv[4 * q + 1] = v.y; hv[4 * q + 2] = v.z; hv[4 * q + 3] = v.w;
                }
                const float o = group_sum<LPR>(d * groups_dot<GPL>(blk, g0, hv, grid_s));
                if (sl == 0) {
                    const uint32_t p = p0 + j0 + jj;
                    outbuf[((size_t)pair_tok[p] * K + pair_k[p]) * H + r0 + rr] = o;
                }
            }
        }
    }
}

template <int GPL>
static rl_status launch_pf32_gateup(const PrefillArgs &a, cudaStream_t s) {
    const size_t sm = gu_smem(a.H);
    rl_status st = allow_smem((const void *)pf32_gateup_kernel<GPL>, sm);
    if (st != RL_OK) return st;
    pf32_gateup_kernel<GPL><<<dim3(a.E, a.I / kPfRows), kPfThreads, sm, s>>>(
        a.xn, a.offs, a.pair_tok, a.pair_k, a.slots, a.codebook, a.hbuf, a.ctrl, a.layer, a.H, a.I, a.K);
    return check_launch("moe_prefill_chunk_f32 gate/up");
}

template <int GPL, int LPR>
static rl_status launch_pf32_down(const PrefillArgs &a, cudaStream_t s) {
    const size_t sm = dn_smem(a.I);
    rl_status st = allow_smem((const void *)pf32_down_kernel<GPL, LPR>, sm);
    if (st != RL_OK) return st;
    pf32_down_kernel<GPL, LPR><<<dim3(a.E, a.H / kPfDownRows), kPfThreads, sm, s>>>(
        a.offs, a.pair_tok, a.pair_k, a.slots, a.codebook, a.hbuf, a.outbuf, a.ctrl, a.layer, a.H, a.I, a.K);
    return check_launch("moe_prefill_chunk_f32 down");
}

}  // namespace rl

using namespace rl;

extern "C" rl_status moe_prefill_chunk_f32(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn,
                                           const uint32_t *offs, const uint32_t *pair_tok, const uint8_t *pair_k,
                                           const uint64_t *slots, const float *weights, const int8_t *codebook,
                                           float *y, int32_t accumulate, int32_t *ctrl, void *ws, size_t ws_bytes,
                                           void *stream) {
    PrefillArgs a;
    rl_status st = prefill_check(shp, layer, T, xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate,
                                 ctrl, ws, ws_bytes, "moe_prefill_chunk_f32", &a);
    if (st != RL_OK || T == 0) return st;
    cudaStream_t s = as_stream(stream);
    switch (a.H) {
        case 256: st = launch_pf32_gateup<1>(a, s); break;
        case 512: st = launch_pf32_gateup<2>(a, s); break;
        case 1024: st = launch_pf32_gateup<4>(a, s); break;
        default: st = launch_pf32_gateup<8>(a, s); break;
    }
    if (st != RL_OK) return st;
    switch (a.I) {
        case 128: st = launch_pf32_down<1, 16>(a, s); break;
        case 256: st = launch_pf32_down<1, 32>(a, s); break;
        case 512: st = launch_pf32_down<2, 32>(a, s); break;
        case 1024: st = launch_pf32_down<4, 32>(a, s); break;
        case 2048: st = launch_pf32_down<8, 32>(a, s); break;
        default: return fail(RL_ERR_UNSUPPORTED, "moe_prefill_chunk_f32: inter=%d", a.I);
    }
    if (st != RL_OK) return st;
    return launch_ordered_sum(a, s);
}
