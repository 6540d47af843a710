// prefill_tc.cu - grouped expert GEMMs of a prefill chunk on the tcgen05 tensor cores.
//
// Red Lite dev20 - batched prompt ingestion, "What changed" item 3: the chunk's routed experts
// run as batched gate/up and down over (expert, token) pairs sorted by expert, then each
// token's top-k outputs are accumulated in router selection order.  Section "dev20d: expert
// kernel layout" decodes each block one 8-value group at a time on another GPU; here the
// decoded weights feed the 5th-generation tensor cores:
//
//   unit = (expert e, token block of <= 128 of its pairs, row tile); one CTA per SM walks the
//   device-built unit list.  Per unit:
//     - one elected thread bulk-copies the unit's quantized weight rows into shared memory
//       (gate/up tile: 64 gate rows + the same 64 up rows, so SwiGLU pairs stay in the CTA;
//       down tile: 128 rows);
//     - K is streamed in chunks of 64: every thread decodes its share of the 128 x 64 A chunk
//       (codebook value with its sign, WITHOUT the block scale: the values are small integers,
//       exact in 16 bits) straight into the canonical K-major core-matrix layout, while
//       cp.async gathers the matching 64 columns of the unit's token rows (B) two chunks ahead;
//     - one thread issues tcgen05.mma (M = 128, N = tokens rounded to 16, K = 16 x 4) into a
//       separate f32 tensor-memory accumulator per 256-value block of the row, and commits to
//       the stage's mbarrier;
//     - epilogue: tcgen05.ld -> registers; the block scales are applied in f32,
//       D[m][n] = sum_b d[m][b] * D_b[m][n]; then h = silu(g) * u (16-bit, pair order) for
//       gate/up, or the f32 per-pair outputs of down, indexed by (token, k) for the combine.
// So the only 16-bit roundings are the activations (x, h).  Operand type T16 is bf16 (the
// default) or f16; both operands of one MMA share it.
#include <algorithm>

#include "prefill_common.cuh"
#include "qdot.cuh"
#include "tc_desc.cuh"

namespace rl {

constexpr int kTcThreads = 256;
constexpr int kNT = 128;         // max tokens per unit
constexpr int kKC = 64;          // K elements per chunk
constexpr int kStageA = 128 * kKC * 2;
constexpr int kStageB = kNT * kKC * 2;
constexpr int kTmemCols = 512;   // per-block accumulators x tokens fill tensor memory at most

// accumulators (256-value blocks) per row of length C, and tokens per unit
__host__ __device__ inline int tc_nblk(int C) { return C >= 256 ? C / 256 : 1; }
__host__ __device__ inline int tc_nt(int C) { return kTmemCols / tc_nblk(C) < kNT ? kTmemCols / tc_nblk(C) : kNT; }
constexpr int kGuRows = 64;      // gate rows (and up rows) per gate/up unit
constexpr int kDnRowsTc = 128;   // down rows per down unit

template <typename T16>
struct TcType;
template <>
struct TcType<__nv_bfloat16> {
    static constexpr uint32_t fmt = 1;
    __device__ static uint32_t bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
    __device__ static uint32_t mul2(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
};
template <>
struct TcType<__half> {
    static constexpr uint32_t fmt = 0;
    __device__ static uint32_t bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
    __device__ static uint32_t mul2(uint32_t a, uint32_t b) {
        __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
};

// codebook as 16-bit pairs of type T16, 8 interleaved copies (see qdot.cuh)
template <typename T16>
__device__ void build_pair_table_t(uint4 *tab, const int8_t *__restrict__ codebook) {
    for (int e = threadIdx.x; e < 256; e += blockDim.x) {
        const uint2 raw = reinterpret_cast<const uint2 *>(codebook)[e];
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t word = p < 2 ? raw.x : raw.y;
            const int g0 = (int8_t)((word >> (16 * (p & 1))) & 0xffu);
            const int g1 = (int8_t)((word >> (16 * (p & 1) + 8)) & 0xffu);
            w[p] = TcType<T16>::bits((float)g0) | (TcType<T16>::bits((float)g1) << 16);
        }
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int c = 0; c < kTabCopies; ++c) tab[e * kTabCopies + ((c + threadIdx.x) & (kTabCopies - 1))] = v;
    }
}

struct TcUnits {   // unit lists in the workspace: [count_gu, count_dn, pad..][gu units][dn units]
    uint32_t *counts, *gu, *dn;
    size_t max_gu, max_dn;
};

__host__ __device__ inline size_t tc_max_units(int P, int E, int nt, int per_block) {
    return ((size_t)P / nt + E) * per_block;
}

// ---- unit lists: per expert ceil(n_e / kNT) token blocks x row tiles -------------------------
// block-wide exclusive scan of one value per thread (blockDim <= 512); returns (prefix, total)
__device__ __forceinline__ uint2 block_scan512(uint32_t v, uint32_t *scan_s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();
    if (lane == 31) scan_s[warp] = incl;
    __syncthreads();
    uint32_t base = 0, total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        if (w < warp) base += scan_s[w];
        total += scan_s[w];
    }
    return make_uint2(base + incl - v, total);
}

// unit = (expert, token block, row tile); token blocks of nt_gu (gate/up) and nt_dn (down)
__global__ void __launch_bounds__(512) tc_units_kernel(const uint32_t *__restrict__ offs, int E, int nt_gu,
                                                       int gu_tiles, int nt_dn, int dn_tiles, uint32_t *counts,
                                                       uint32_t *gu, uint32_t *dn, const int32_t *ctrl, int layer) {
    __shared__ uint32_t scan_s[16];
    if (ld_ctrl(ctrl) <= layer) return;
    const int e = threadIdx.x;
    const uint32_t n = e < E ? offs[e + 1] - offs[e] : 0u;
    const uint32_t nbg = (n + nt_gu - 1) / nt_gu, nbd = (n + nt_dn - 1) / nt_dn;
    const uint2 sg = block_scan512(nbg, scan_s);
    const uint2 sd = block_scan512(nbd, scan_s);
    for (uint32_t tb = 0; tb < nbg; ++tb)
        for (int mt = 0; mt < gu_tiles; ++mt) gu[(sg.x + tb) * gu_tiles + mt] = e | (tb << 10) | ((uint32_t)mt << 20);
    for (uint32_t tb = 0; tb < nbd; ++tb)
        for (int mt = 0; mt < dn_tiles; ++mt) dn[(sd.x + tb) * dn_tiles + mt] = e | (tb << 10) | ((uint32_t)mt << 20);
    if (e == 0) {
        counts[0] = sg.y * gu_tiles;
        counts[1] = sd.y * dn_tiles;
    }
}

template <typename T16>
__global__ void __launch_bounds__(256) tc_convert_kernel(const float *__restrict__ x, uint16_t *__restrict__ xb,
                                                         size_t n, const int32_t *ctrl, int layer) {
    if (ld_ctrl(ctrl) <= layer) return;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        xb[i] = (uint16_t)TcType<T16>::bits(x[i]);
}

// ---- the grouped GEMM -------------------------------------------------------------------------
struct TcLayout {
    size_t raw, total;   // bytes of the raw quantized rows of one unit; total shared memory
    __host__ __device__ TcLayout(int MODE, int H, int I) {
        raw = MODE == 0 ? 2 * matrix_bytes(kGuRows, H) : matrix_bytes(kDnRowsTc, I);
        raw = align_up(raw, 128);
        total = 1024 + kTabBytes + raw + 2 * kStageA + 2 * kStageB;
    }
};

// MODE 0: gate/up -> hb (16-bit h, pair order).  MODE 1: down -> outbuf (f32, (token, k) order).
template <typename T16, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(PrefillArgs a, TcUnits U) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *raw_bar = reinterpret_cast<uint64_t *>(smem);       // bulk copy of a unit's rows
    uint64_t *mma_bar = raw_bar + 1;                              // [2] one per stage
    uint64_t *done_bar = raw_bar + 3;                             // a unit's MMAs complete
    uint64_t *fin_bar = raw_bar + 4;                              // drain before TMEM release
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(smem + 64);
    uint32_t *tok_s = reinterpret_cast<uint32_t *>(smem + 128);   // [kNT] token of each pair
    uint8_t *k_s = smem + 128 + 4 * kNT;                          // [kNT] k of each pair
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 1024);
    const TcLayout lay(MODE, a.H, a.I);
    uint8_t *raw = smem + 1024 + kTabBytes;
    uint8_t *stA = raw + lay.raw;                                 // [2][kStageA]
    uint8_t *stB = stA + 2 * kStageA;                             // [2][kStageB]
    float *u_s = reinterpret_cast<float *>(stA);                  // epilogue exchange (gate/up)

    if (ld_ctrl(a.ctrl) <= a.layer) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&raw_bar[i], 1);
        fence_mbar_init();
    }
    const int C = MODE == 0 ? a.H : a.I;                 // K of this GEMM (row length)
    const int nblk = tc_nblk(C), nt = tc_nt(C);
    const uint32_t tcols = (uint32_t)(nblk * nt);        // 128, 256 or 512
    if (warp == 0) {
        tc::tmem_alloc(tmem_s, tcols);
        tc::tmem_relinquish();
    }
    build_pair_table_t<T16>(tab, a.codebook);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_s;

    const int nch = C / kKC;
    const size_t rowb_q = matrix_bytes(1, a.H);          // bytes of an H-wide row (gate/up)
    const size_t matb = matrix_bytes(a.I, a.H);
    const uint32_t count = __ldcg(&U.counts[MODE]);
    const uint32_t *units = MODE == 0 ? U.gu : U.dn;
    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
    uint32_t gc = 0, nunits = 0;
    bool failed = false;

    for (uint32_t ui = blockIdx.x; ui < count; ui += gridDim.x) {
        const uint32_t uw = __ldcg(&units[ui]);
        const int e = uw & 1023, tb = (uw >> 10) & 1023, mt = uw >> 20;
        const uint32_t pe0 = __ldcg(&a.offs[e]), pe1 = __ldcg(&a.offs[e + 1]);
        const uint32_t p_lo = pe0 + tb * nt;
        const int nvalid = (int)min((uint32_t)nt, pe1 - p_lo);
        const int npad = (nvalid + 15) & ~15;
        if (tid < nvalid) {
            tok_s[tid] = __ldcg(&a.pair_tok[p_lo + tid]);
            k_s[tid] = __ldcg(&a.pair_k[p_lo + tid]);
        }
        __syncthreads();
        // the unit's expert record
        const uint64_t slot = __ldcg(&a.slots[(size_t)tok_s[0] * a.K + k_s[0]]);
        const bool bad = slot == 0 || (slot & 15);
        if (bad) {
            if (tid == 0) dev_error(a.ctrl, slot == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
            __syncthreads();
            continue;
        }
        const uint8_t *rec = reinterpret_cast<const uint8_t *>(slot);
        if (tid == 0) {
            if (MODE == 0) {
                const uint32_t b = (uint32_t)(kGuRows * rowb_q);
                const uint8_t *g = rec + (size_t)mt * kGuRows * rowb_q;
                mbar_arrive_expect_tx(raw_bar, 2 * b);
                bulk_g2s(raw, g, b, raw_bar);
                bulk_g2s(raw + b, g + matb, b, raw_bar);
            } else {
                const uint32_t b = (uint32_t)matrix_bytes(kDnRowsTc, a.I);
                mbar_arrive_expect_tx(raw_bar, b);
                bulk_g2s(raw, rec + 2 * matb + matrix_bytes(mt * kDnRowsTc, a.I), b, raw_bar);
            }
        }
        // B rows of chunk c go to stage (gc + c) & 1
        auto issue_b = [&](int c, uint8_t *dstB) {
            for (int i = tid; i < npad * 8; i += kTcThreads) {
                const int n = i % npad, j = i / npad;
                uint8_t *d = dstB + ((n >> 3) * 8 + j) * 128 + (n & 7) * 16;
                if (n < nvalid) {
                    const uint16_t *src = MODE == 0
                                              ? a.xb16 + (size_t)tok_s[n] * a.H + c * kKC + j * 8
                                              : a.hb16 + (size_t)(p_lo + n) * a.I + c * kKC + j * 8;
                    tc::cp_async16(d, src);
                } else {
                    *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc::cp_async_commit();
        };
        issue_b(0, stB + (gc & 1) * kStageB);
        failed |= !mbar_wait(raw_bar, nunits & 1);
        if ((failed = __syncthreads_or(failed) != 0)) break;
        const uint32_t idesc = tc::instr_desc(TcType<T16>::fmt, 128, npad);
        for (int c = 0; c < nch; ++c, ++gc) {
            const int s = gc & 1;
            // the other stage was last read by the MMAs of chunk gc - 1
            if (gc >= 1) failed |= !mbar_wait(&mma_bar[(gc - 1) & 1], ((gc - 1) >> 1) & 1);
            if (c + 1 < nch) issue_b(c + 1, stB + (s ^ 1) * kStageB);
            // decode this thread's items of the 128 x 64 A chunk into stage s
            uint8_t *dA = stA + s * kStageA;
            for (int i = tid; i < 128 * 8; i += kTcThreads) {
                const int row = i & 127, j = i >> 7;
                int r = row;
                const uint8_t *rb = raw;
                if (MODE == 0 && row >= kGuRows) {  // rows 64..127: the up matrix
                    r = row - kGuRows;
                    rb = raw + matrix_bytes(kGuRows, a.H);
                }
                const int G = r * (C / 8) + c * 8 + j;  // flat group index inside the raw rows
                const uint8_t *blk = rb + (G >> 5) * kBlockBytes;
                const uint32_t gs = *reinterpret_cast<const uint16_t *>(blk + 2 + 2 * (G & 31));
                const uint4 q = tabc[(gs & 0xffu) * kTabCopies];
                const uint32_t sgn = (gs >> 8) & 0xffu;
                const uint32_t s2 = sgn | ((sgn << 15) & 0x007f0000u);
                uint4 v;  // +-codebook value, exact in 16 bits; the block scale is applied later
                v.x = q.x ^ ((s2 << 15) & 0x80008000u);
                v.y = q.y ^ ((s2 << 13) & 0x80008000u);
                v.z = q.z ^ ((s2 << 11) & 0x80008000u);
                v.w = q.w ^ ((s2 << 9) & 0x80008000u);
                *reinterpret_cast<uint4 *>(dA + ((row >> 3) * 8 + j) * 128 + (row & 7) * 16) = v;
            }
            if (c + 1 < nch) tc::cp_async_wait<1>();
            else tc::cp_async_wait<0>();
            fence_proxy_async_smem();
            if ((failed = __syncthreads_or(failed) != 0)) break;
            if (tid == 0) {
                tc::fence_after();
                const uint32_t aB = tc::s_addr(dA), bB = tc::s_addr(stB + s * kStageB);
                // chunk c lies in 256-value block c * kKC / 256 of the row: its own accumulator
                const int blk = nblk == 1 ? 0 : (c * kKC) / 256;
                const bool first = (c * kKC) % 256 == 0 || nblk == 1 && c == 0;
#pragma unroll
                for (int kk = 0; kk < kKC / 16; ++kk)
                    tc::mma_f16(tmem + (uint32_t)(blk * nt), tc::smem_desc(aB + kk * 256, 128, 1024),
                                tc::smem_desc(bB + kk * 256, 128, 1024), idesc, (first && kk == 0) ? 0u : 1u);
                tc::commit(&mma_bar[s]);
            }
        }
        if (failed) break;
        if (tid == 0) tc::commit(done_bar);
        failed |= !mbar_wait(done_bar, nunits & 1);
        ++nunits;
        if ((failed = __syncthreads_or(failed) != 0)) break;
        tc::fence_after();
        // ---- epilogue: warps 0..3 own TMEM lanes 0..127 = A rows ---------------------------------
        // D[row][n] = sum_b d[row][b] * D_b[row][n], with D_b at TMEM columns b * nt + n
        if (warp < 4) {
            const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
            int r = tid;                              // row inside this unit's raw rows
            const uint8_t *rb = raw;
            if (MODE == 0 && tid >= kGuRows) {
                r = tid - kGuRows;
                rb = raw + matrix_bytes(kGuRows, a.H);
            }
            float dsc[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int G = r * (C / 8) + (nblk == 1 ? 0 : 32 * b);
                dsc[b] = b < nblk ? fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(rb + (G >> 5) * kBlockBytes))
                                  : 0.f;
            }
            auto scaled16 = [&](int c0, float (&acc)[16]) {
#pragma unroll
                for (int q = 0; q < 16; ++q) acc[q] = 0.f;
                for (int b = 0; b < nblk; ++b) {
                    uint32_t v[16];
                    tc::ld16(trow + (uint32_t)(b * nt + c0), v);
                    tc::ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) acc[q] = fmaf(dsc[b], __uint_as_float(v[q]), acc[q]);
                }
            };
            if (MODE == 0) {
                if (warp >= 2) {  // up rows: park u in shared memory
                    for (int c0 = 0; c0 < npad; c0 += 16) {
                        float acc[16];
                        scaled16(c0, acc);
#pragma unroll
                        for (int q = 0; q < 16; ++q) u_s[r * kNT + c0 + q] = acc[q];
                    }
                }
            } else {
                const int orow = mt * kDnRowsTc + tid;  // output row of H
                for (int c0 = 0; c0 < npad; c0 += 16) {
                    float acc[16];
                    scaled16(c0, acc);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int n = c0 + q;
                        if (n < nvalid) a.outbuf[((size_t)tok_s[n] * a.K + k_s[n]) * a.H + orow] = acc[q];
                    }
                }
            }
            if (MODE == 0) asm volatile("bar.sync 1, 128;" ::: "memory");  // up rows parked (warps 0-3 only)
            if (MODE == 0 && warp < 2) {  // gate rows: h = silu(g) * u
                uint16_t *hb = a.hb16 + (size_t)p_lo * a.I + (size_t)mt * kGuRows + r;
                for (int c0 = 0; c0 < npad; c0 += 16) {
                    float acc[16];
                    scaled16(c0, acc);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int n = c0 + q;
                        if (n < nvalid) hb[(size_t)n * a.I] = (uint16_t)TcType<T16>::bits(silu(acc[q]) * u_s[r * kNT + n]);
                    }
                }
            }
        }
        tc::fence_before();
        __syncthreads();
    }
    if (failed && tid == 0) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);
    // drain every tcgen05 operation this CTA issued, then release tensor memory
    if (tid == 0) {
        tc::commit(fin_bar);
        mbar_wait(fin_bar, 0);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, tcols);
}

template <typename T16>
static rl_status run_tc(const PrefillArgs &a0, cudaStream_t s) {
    PrefillArgs a = a0;
    const int P = a.P, E = a.E;
    const int gu_tiles = a.I / kGuRows, dn_tiles = a.H / kDnRowsTc;
    TcUnits U;
    uint8_t *ub = reinterpret_cast<uint8_t *>(a.units);
    U.counts = reinterpret_cast<uint32_t *>(ub);
    const int nt_gu = tc_nt(a.H), nt_dn = tc_nt(a.I);
    U.max_gu = tc_max_units(P, E, nt_gu, gu_tiles);
    U.max_dn = tc_max_units(P, E, nt_dn, dn_tiles);
    U.gu = reinterpret_cast<uint32_t *>(ub + 256);
    U.dn = U.gu + U.max_gu;
    const size_t n = (size_t)a.T * a.H;
    tc_convert_kernel<T16><<<(int)std::min<size_t>((n + 255) / 256, 4096), 256, 0, s>>>(a.xn, a.xb16, n, a.ctrl,
                                                                                       a.layer);
    tc_units_kernel<<<1, 512, 0, s>>>(a.offs, E, nt_gu, gu_tiles, nt_dn, dn_tiles, U.counts, U.gu, U.dn, a.ctrl,
                                      a.layer);
    rl_status st = check_launch("moe_prefill_chunk setup");
    if (st != RL_OK) return st;
    const int sms = sm_count();
    {
        const TcLayout lay(0, a.H, a.I);
        st = allow_smem((const void *)tc_gemm_kernel<T16, 0>, lay.total);
        if (st != RL_OK) return st;
        tc_gemm_kernel<T16, 0><<<(int)std::min<size_t>(sms, U.max_gu), kTcThreads, lay.total, s>>>(a, U);
        st = check_launch("moe_prefill_chunk gate/up");
        if (st != RL_OK) return st;
    }
    {
        const TcLayout lay(1, a.H, a.I);
        st = allow_smem((const void *)tc_gemm_kernel<T16, 1>, lay.total);
        if (st != RL_OK) return st;
        tc_gemm_kernel<T16, 1><<<(int)std::min<size_t>(sms, U.max_dn), kTcThreads, lay.total, s>>>(a, U);
        st = check_launch("moe_prefill_chunk down");
        if (st != RL_OK) return st;
    }
    return launch_ordered_sum(a, s);
}

}  // namespace rl

using namespace rl;

extern "C" rl_status moe_prefill_chunk(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn,
                                       const uint32_t *offs, const uint32_t *pair_tok, const uint8_t *pair_k,
                                       const uint64_t *slots, const float *weights, const int8_t *codebook,
                                       float *y, int32_t accumulate, int32_t *ctrl, void *ws, size_t ws_bytes,
                                       void *stream) {
    PrefillArgs a;
    rl_status st = prefill_check(shp, layer, T, xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate,
                                 ctrl, ws, ws_bytes, "moe_prefill_chunk", &a);
    if (st != RL_OK || T == 0) return st;
    return run_tc<__nv_bfloat16>(a, as_stream(stream));
}
