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

constexpr int kNT = 128;         // max tokens per unit
#ifndef RL_TC_KC
#define RL_TC_KC 64
#endif
constexpr int kKC = RL_TC_KC;    // K elements per chunk
constexpr int kKG = kKC / 8;     // 16-byte core-matrix columns (8 values) per chunk

// accumulators (256-value blocks) per row of length C
__host__ __device__ inline int tc_nblk(int C) { return C >= 256 ? C / 256 : 1; }
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

// ---- the grouped GEMM: a warp-specialised pipeline -------------------------------------------
// Warp roles (18 warps):
//   0-11  producers: for every 64-wide K chunk of a unit, gather the unit's token rows of the
//         B operand (16-bit activations) and decode the 128 x 64 A chunk from the quantized rows
//         into one stage of a ring (canonical K-major core-matrix layout), then arrive on the
//         stage's "full" barrier;
//   12    MMA issuer (lane 0): per chunk, waits "full", issues the tcgen05.mma of the chunk into
//         the unit's tensor-memory accumulators and commits to the stage's "empty" barrier;
//         after a unit's last chunk, commits to the accumulator's "full" barrier;
//   13    loader: stages the next unit's token list and bulk-copies its quantized rows into the
//         other of two raw buffers;
//   14-17 epilogue: the four TMEM lane quadrants (warp w reads lanes 32 (w % 4) ...); applies the
//         block scales and writes h (gate/up) or the per-pair outputs (down), then releases the
//         accumulator and the raw buffer.
// The accumulators (one per 256-value block, nt tokens wide) are double-buffered in tensor
// memory, so a unit's epilogue overlaps the next unit's MMAs; the raw rows are double-buffered
// so the next unit's copy overlaps the current unit.  Every wait is bounded; a timeout sets a
// shared abort flag and every role leaves its loop.
constexpr int kTcProducers = 12;
constexpr int kTcMmaWarp = 12;
constexpr int kTcLoadWarp = 13;
constexpr int kTcEpiWarp0 = 14;
constexpr int kTcThreads2 = 18 * 32;
constexpr int kTcPT = kTcProducers * 32;              // producer threads
constexpr int kTcBMax = (kNT * kKG + kTcPT - 1) / kTcPT;  // B pieces per producer thread and chunk
constexpr int kTcAItems = (128 * kKG + kTcPT - 1) / kTcPT;
#ifndef RL_TC_STAGES
#define RL_TC_STAGES 2
#endif
constexpr int kTcStages = RL_TC_STAGES;

// tokens per unit when the accumulators are double-buffered: 2 x nblk x nt <= 512 columns
__host__ __device__ inline int tc_nt2(int C) { return 256 / tc_nblk(C) < kNT ? 256 / tc_nblk(C) : kNT; }

struct TcMeta {        // one unit, staged by the loader
    int e, mt, nvalid, npad;
    uint32_t p_lo;
    uint32_t tok[kNT];
    uint8_t k[kNT];
};

struct TcLayout {
    size_t raw, stA, stB, o_meta, o_raw, o_st, o_u, total;
    __host__ __device__ TcLayout(int MODE, int H, int I) {
        raw = align_up(MODE == 0 ? 2 * matrix_bytes(kGuRows, H) : matrix_bytes(kDnRowsTc, I), 128);
        const int nt = tc_nt2(MODE == 0 ? H : I);
        stA = 128 * kKC * 2;
        stB = (size_t)nt * kKC * 2;
        o_meta = 1024 + kTabBytes;
        o_raw = align_up(o_meta + 2 * sizeof(TcMeta), 128);
        o_st = o_raw + 2 * raw;
        o_u = o_st + kTcStages * (stA + stB);
        total = o_u + (MODE == 0 ? (size_t)kGuRows * nt * sizeof(float) : 0);
    }
};

// MODE 0: gate/up -> hb (16-bit h, pair order).  MODE 1: down -> outbuf (f32, (token, k) order).
template <typename T16, int MODE>
__global__ void __launch_bounds__(kTcThreads2, 1) tc_gemm_kernel(PrefillArgs a, TcUnits U) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint64_t *raw_full = bars, *raw_empty = bars + 2;          // [2] each
    uint64_t *acc_full = bars + 4, *acc_empty = bars + 6;      // [2] each
    uint64_t *st_full = bars + 8, *st_empty = bars + 8 + kTcStages;
    uint64_t *fin_bar = bars + 8 + 2 * kTcStages;
    uint64_t *ex_full = fin_bar + 1, *ex_empty = fin_bar + 2;  // gate/up epilogue: u parked / consumed
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(smem + 256);
    int *abort_s = reinterpret_cast<int *>(smem + 260);
    uint4 *tab = reinterpret_cast<uint4 *>(smem + 1024);
    const TcLayout lay(MODE, a.H, a.I);
    TcMeta *meta = reinterpret_cast<TcMeta *>(smem + lay.o_meta);
    uint8_t *rawb = smem + lay.o_raw;                            // [2][lay.raw]
    uint8_t *stg = smem + lay.o_st;                              // [kTcStages][stA + stB]
    float *u_s = reinterpret_cast<float *>(smem + lay.o_u);      // [kGuRows][nt] (gate/up)

    if (ld_ctrl(a.ctrl) <= a.layer) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = MODE == 0 ? a.H : a.I;  // K of this GEMM (row length)
    const int nblk = tc_nblk(C), nt = tc_nt2(C);
    const int nch = C / kKC;
    const uint32_t acc_cols = (uint32_t)(nblk * nt);  // one accumulator set; two are allocated
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&bars[i], (i >= 2 && i < 4) ? kTcProducers + 4 : (i >= 6 ? 4 : 1));
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&st_full[i], kTcProducers);
            mbar_init(&st_empty[i], 1);
        }
        mbar_init(fin_bar, 1);
        mbar_init(ex_full, 2);   // the two up-row warps
        mbar_init(ex_empty, 2);  // the two gate-row warps
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_s, 512);
        tc::tmem_relinquish();
    }
    build_pair_table_t<T16>(tab, a.codebook);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_s;
    const uint32_t count = __ldcg(&U.counts[MODE]);
    const uint32_t *units = MODE == 0 ? U.gu : U.dn;
    const uint32_t nmine = count > blockIdx.x ? (count - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
    const size_t rowb_q = matrix_bytes(1, a.H);  // bytes of an H-wide row (gate/up)
    const size_t matb = matrix_bytes(a.I, a.H);
    bool failed = false;
    // whole warp; bounded; sets the abort flag.  The per-chunk hand-offs between producers and
    // the MMA issuer spin on test_wait (a suspended try_wait wakes too late for them); the
    // long waits (a whole unit) suspend, so that waiting warps leave the issue slots free.
    auto wait_spin = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_spin_warp(bar, parity)) {
            if (lane == 0) atomicExch(abort_s, 1);
            failed = true;
        }
        return !failed;
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_wait_warp(bar, parity)) {
            if (lane == 0) atomicExch(abort_s, 1);
            failed = true;
        }
        return !failed;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(abort_s) != 0; };

    if (warp == kTcLoadWarp) {
        // ---------------- loader ----------------
        uint32_t issued = 0;
        for (uint32_t k = 0; k < nmine && !failed && !aborted(); ++k) {
            const int rb = k & 1;
            if (k >= 2 && !wait(&raw_empty[rb], ((k >> 1) - 1) & 1)) break;
            const uint32_t uw = __ldcg(&units[blockIdx.x + k * gridDim.x]);
            const int e = uw & 1023, tb = (uw >> 10) & 1023, mt = uw >> 20;
            const uint32_t pe0 = __ldcg(&a.offs[e]), pe1 = __ldcg(&a.offs[e + 1]);
            const uint32_t p_lo = pe0 + tb * nt;
            const int nvalid = (int)min((uint32_t)nt, pe1 - p_lo);
            TcMeta &m = meta[rb];
            for (int i = lane; i < nvalid; i += 32) {
                m.tok[i] = __ldcg(&a.pair_tok[p_lo + i]);
                m.k[i] = __ldcg(&a.pair_k[p_lo + i]);
            }
            if (lane == 0) {
                m.e = e;
                m.mt = mt;
                m.nvalid = nvalid;
                m.npad = (nvalid + 15) & ~15;
                m.p_lo = p_lo;
            }
            __syncwarp();
            if (lane == 0) {
                const uint64_t slot = __ldcg(&a.slots[(size_t)m.tok[0] * a.K + m.k[0]]);
                if (slot == 0 || (slot & 15)) {
                    // nothing is copied: the unit's outputs are garbage and the host sees the flag
                    dev_error(a.ctrl, slot == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
                    mbar_arrive(&raw_full[rb]);
                } else {
                    const uint8_t *rec = reinterpret_cast<const uint8_t *>(slot);
                    uint8_t *dst = rawb + rb * lay.raw;
                    if (MODE == 0) {
                        const uint32_t b = (uint32_t)(kGuRows * rowb_q);
                        const uint8_t *g = rec + (size_t)mt * kGuRows * rowb_q;
                        mbar_arrive_expect_tx(&raw_full[rb], 2 * b);
                        bulk_g2s(dst, g, b, &raw_full[rb]);
                        bulk_g2s(dst + b, g + matb, b, &raw_full[rb]);
                    } else {
                        const uint32_t b = (uint32_t)matrix_bytes(kDnRowsTc, a.I);
                        mbar_arrive_expect_tx(&raw_full[rb], b);
                        bulk_g2s(dst, rec + 2 * matb + matrix_bytes(mt * kDnRowsTc, a.I), b, &raw_full[rb]);
                    }
                }
            }
            __syncwarp();
            issued = k + 1;
        }
        // every copy this warp issued must have landed before the CTA may exit
        for (uint32_t k = issued >= 2 ? issued - 2 : 0; k < issued; ++k) mbar_wait_warp(&raw_full[k & 1], (k >> 1) & 1);
    } else if (warp < kTcProducers) {
        // ---------------- producers ----------------
        const uint4 *tabc = tab + (lane & (kTabCopies - 1));
        uint32_t g = 0;  // chunk counter over all units
        for (uint32_t k = 0; k < nmine && !failed; ++k) {
            const int rb = k & 1;
            if (!wait(&raw_full[rb], (k >> 1) & 1)) break;
            const TcMeta &m = meta[rb];
            const int nvalid = m.nvalid, npad = m.npad;
            const uint8_t *raw = rawb + rb * lay.raw;
            // B pieces of chunk c for this thread: i = tid + kTcPT * t < npad * 8
            auto load_b = [&](int c, uint4 (&bv)[kTcBMax]) {
#pragma unroll
                for (int t = 0; t < kTcBMax; ++t) {
                    const int i = tid + kTcPT * t;
                    const int n = i % npad, j = i / npad;
                    bv[t] = make_uint4(0u, 0u, 0u, 0u);
                    if (i < npad * kKG && n < nvalid) {
                        const uint16_t *src = MODE == 0 ? a.xb16 + (size_t)m.tok[n] * a.H + c * kKC + j * 8
                                                        : a.hb16 + (size_t)(m.p_lo + n) * a.I + c * kKC + j * 8;
                        bv[t] = __ldg(reinterpret_cast<const uint4 *>(src));
                    }
                }
            };
            uint4 bv[kTcBMax];
            load_b(0, bv);
            for (int c = 0; c < nch && !failed; ++c, ++g) {
                const int s = g % kTcStages;
                if (g >= (uint32_t)kTcStages && !wait_spin(&st_empty[s], ((g / kTcStages) - 1) & 1)) break;
                if (aborted()) { failed = true; break; }
                uint8_t *dA = stg + s * (lay.stA + lay.stB);
                uint8_t *dB = dA + lay.stA;
                // B of this chunk (loaded one chunk ahead), then the loads of the next chunk
#pragma unroll
                for (int t = 0; t < kTcBMax; ++t) {
                    const int i = tid + kTcPT * t;
                    if (i < npad * kKG) {
                        const int n = i % npad, j = i / npad;
                        *reinterpret_cast<uint4 *>(dB + ((n >> 3) * kKG + j) * 128 + (n & 7) * 16) = bv[t];
                    }
                }
                if (c + 1 < nch) load_b(c + 1, bv);
                // A: the 128 x 64 chunk as +-codebook values (exact in 16 bits), no block scale;
                // all loads of the thread's items first, then the stores
                uint32_t gs[kTcAItems];
                int row_[kTcAItems], j_[kTcAItems];
#pragma unroll
                for (int t = 0; t < kTcAItems; ++t) {
                    const int i = tid + kTcPT * t;
                    const int row = i & 127, j = i >> 7;
                    row_[t] = row;
                    j_[t] = j;
                    gs[t] = 0;
                    if (i < 128 * kKG) {
                        int r = row;
                        const uint8_t *rb_ = raw;
                        if (MODE == 0 && row >= kGuRows) {  // rows 64..127: the up matrix
                            r = row - kGuRows;
                            rb_ = raw + matrix_bytes(kGuRows, a.H);
                        }
                        const int G = r * (C / 8) + c * kKG + j;  // flat group index inside the raw rows
                        gs[t] = *reinterpret_cast<const uint16_t *>(rb_ + (G >> 5) * kBlockBytes + 2 + 2 * (G & 31));
                    }
                }
                uint4 q[kTcAItems];
#pragma unroll
                for (int t = 0; t < kTcAItems; ++t) q[t] = tabc[(gs[t] & 0xffu) * kTabCopies];
#pragma unroll
                for (int t = 0; t < kTcAItems; ++t) {
                    if (tid + kTcPT * t < 128 * kKG) {
                        const uint32_t sgn = (gs[t] >> 8) & 0xffu;
                        const uint32_t s2 = sgn | ((sgn << 15) & 0x007f0000u);
                        uint4 v;
                        v.x = q[t].x ^ ((s2 << 15) & 0x80008000u);
                        v.y = q[t].y ^ ((s2 << 13) & 0x80008000u);
                        v.z = q[t].z ^ ((s2 << 11) & 0x80008000u);
                        v.w = q[t].w ^ ((s2 << 9) & 0x80008000u);
                        const int row = row_[t];
                        *reinterpret_cast<uint4 *>(dA + ((row >> 3) * kKG + j_[t]) * 128 + (row & 7) * 16) = v;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st_full[s]);
            }
            if (failed) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[rb]);
        }
    } else if (warp == kTcMmaWarp) {
        // ---------------- MMA issuer ----------------
        uint32_t g = 0;
        for (uint32_t k = 0; k < nmine && !failed; ++k) {
            const int ab = k & 1;
            if (k >= 2 && !wait(&acc_empty[ab], ((k >> 1) - 1) & 1)) break;
            for (int c = 0; c < nch; ++c, ++g) {
                const int s = g % kTcStages;
                if (!wait_spin(&st_full[s], (g / kTcStages) & 1)) break;
                if (lane == 0) {
                    tc::fence_after();
                    const int npad = meta[k & 1].npad;
                    const uint32_t idesc = tc::instr_desc(TcType<T16>::fmt, 128, npad);
                    const uint8_t *dA = stg + s * (lay.stA + lay.stB);
                    const uint32_t aB = tc::s_addr(dA), bB = tc::s_addr(dA + lay.stA);
                    const int blk = nblk == 1 ? 0 : (c * kKC) / 256;
                    const bool first = nblk == 1 ? c == 0 : (c * kKC) % 256 == 0;
                    const uint32_t d = tmem + (uint32_t)(ab * acc_cols + blk * nt);
#pragma unroll
                    for (int kk = 0; kk < kKC / 16; ++kk)
                        tc::mma_f16(d, tc::smem_desc(aB + kk * 256, 128, kKG * 128),
                                    tc::smem_desc(bB + kk * 256, 128, kKG * 128), idesc, (first && kk == 0) ? 0u : 1u);
                    tc::commit(&st_empty[s]);
                    if (c == nch - 1) tc::commit(&acc_full[ab]);
                }
                __syncwarp();
            }
        }
    } else if (warp >= kTcEpiWarp0) {
        // ---------------- epilogue ----------------
        const int quad = warp & 3;                 // TMEM lanes 32 quad .. 32 quad + 31 = A rows
        const int row = quad * 32 + lane;
        for (uint32_t k = 0; k < nmine && !failed; ++k) {
            const int ab = k & 1, rb = k & 1;
            if (!wait(&acc_full[ab], (k >> 1) & 1)) break;
            tc::fence_after();
            const TcMeta &m = meta[rb];
            const int nvalid = m.nvalid, npad = m.npad, mt = m.mt;
            const uint8_t *raw = rawb + rb * lay.raw;
            int r = row;
            const uint8_t *rr = raw;
            if (MODE == 0 && row >= kGuRows) {
                r = row - kGuRows;
                rr = raw + matrix_bytes(kGuRows, a.H);
            }
            float dsc[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int G = r * (C / 8) + (nblk == 1 ? 0 : 32 * b);
                dsc[b] = b < nblk ? fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(rr + (G >> 5) * kBlockBytes))
                                  : 0.f;
            }
            const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(ab * acc_cols);
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
                if (row >= kGuRows) {  // up rows: park u once the gate rows have used the last one
                    if (k >= 1 && !wait(ex_empty, (k - 1) & 1)) break;
                    for (int c0 = 0; c0 < npad; c0 += 16) {
                        float acc[16];
                        scaled16(c0, acc);
#pragma unroll
                        for (int q = 0; q < 16; ++q) u_s[r * nt + c0 + q] = acc[q];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ex_full);
                } else {               // gate rows: h = silu(g) * u
                    if (!wait(ex_full, k & 1)) break;
                    uint16_t *hb = a.hb16 + (size_t)m.p_lo * a.I + (size_t)mt * kGuRows + r;
                    for (int c0 = 0; c0 < npad; c0 += 16) {
                        float acc[16];
                        scaled16(c0, acc);
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int n = c0 + q;
                            if (n < nvalid) hb[(size_t)n * a.I] = (uint16_t)TcType<T16>::bits(silu(acc[q]) * u_s[r * nt + n]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ex_empty);
                }
            } else {
                const int orow = mt * kDnRowsTc + row;  // output row of H
                for (int c0 = 0; c0 < npad; c0 += 16) {
                    float acc[16];
                    scaled16(c0, acc);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int n = c0 + q;
                        if (n < nvalid) a.outbuf[((size_t)m.tok[n] * a.K + m.k[n]) * a.H + orow] = acc[q];
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[ab]);
                mbar_arrive(&raw_empty[rb]);
            }
        }
    }
    if (failed && lane == 0) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);
    // drain every tcgen05 operation this CTA issued, then release tensor memory
    __syncthreads();
    if (tid == kTcMmaWarp * 32) {
        tc::commit(fin_bar);
        if (!mbar_wait(fin_bar, 0)) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);  // the drain did not finish
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <typename T16>
static rl_status run_tc(const PrefillArgs &a0, cudaStream_t s) {
    PrefillArgs a = a0;
    const int P = a.P, E = a.E;
    const int gu_tiles = a.I / kGuRows, dn_tiles = a.H / kDnRowsTc;
    TcUnits U;
    uint8_t *ub = reinterpret_cast<uint8_t *>(a.units);
    U.counts = reinterpret_cast<uint32_t *>(ub);
    const int nt_gu = tc_nt2(a.H), nt_dn = tc_nt2(a.I);
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
        tc_gemm_kernel<T16, 0><<<(int)std::min<size_t>(sms, U.max_gu), kTcThreads2, lay.total, s>>>(a, U);
        st = check_launch("moe_prefill_chunk gate/up");
        if (st != RL_OK) return st;
    }
    {
        const TcLayout lay(1, a.H, a.I);
        st = allow_smem((const void *)tc_gemm_kernel<T16, 1>, lay.total);
        if (st != RL_OK) return st;
        tc_gemm_kernel<T16, 1><<<(int)std::min<size_t>(sms, U.max_dn), kTcThreads2, lay.total, s>>>(a, U);
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
