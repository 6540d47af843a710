// prefill_tc.cu - grouped expert GEMMs of a prefill chunk on the tcgen05 tensor cores.
//
// Red Lite dev20 - batched prompt ingestion, "What changed" item 3: the chunk's routed experts
// run as batched gate/up and down over (expert, token) pairs sorted by expert, then each
// token's top-k outputs are accumulated in router selection order; a plan covers at most the
// 512 experts of a layer.  Section "dev20d: expert kernel layout" decodes each block one
// 8-value group at a time on another GPU; here the decoded weights feed the 5th-generation
// tensor cores:
//
//   unit = (expert e, token block of <= 128 of its pairs, row tile of 128 weight rows).  The
//   A operand (weights) is decoded from the quantized rows straight into TENSOR MEMORY by the
//   producer warps (tcgen05.st: lane m = weight row m), so the decoded weights never pass
//   through shared memory; the B operand (the unit's activations, 16-bit, pair order) arrives
//   by TMA tensor copies with the 128-byte swizzle; one thread issues
//   tcgen05.mma (A from tensor memory, B from shared memory, f32 accumulator in tensor memory).
//
// Operands are IEEE half precision: a weight is d * codebook[idx][j] * (+-1) rounded once to
// f16 (the product of the f16 scale and the small integer needs up to 17 bits; f16 keeps 11),
// the activations x and h are rounded to f16.  The f32 accumulator sees every K term.
//
// One thread issuing MMAs waits ~54 cycles per M = 128, K = 16 MMA whatever N (measured on
// GB300), while at N = 16 the tensor pipe needs ~8: a unit of at most 64 tokens therefore has
// two issuers, one per producer set, each summing its half of the K steps into an accumulator
// of its own (the epilogue adds the two); a larger unit keeps the pipe busy with one issuer.
//
// Weights are the same for every token of a unit, so a heavy expert (many tokens, the Zipf
// head of a skewed chunk) decodes its rows once per 128 tokens; the unit list puts the full
// 128-token blocks first and the work is taken from a global counter, so the heavy units start
// first and the light ones fill in behind them.
#include <algorithm>

#include "prefill_common.cuh"
#include "qdot.cuh"
#include "tc_desc.cuh"

namespace rl {

// L2 eviction priorities for the copies below: data read once leaves first, data read again
// (by other CTAs or later units) stays longest
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

constexpr int kNT = 128;        // tokens (pairs) per unit, the MMA's N at most
constexpr int kTcRows = 128;    // weight rows per unit: the MMA's M (gate/up: 64 gate + 64 up rows)
constexpr int kGuUnits = 64;    // hidden units per gate/up unit
constexpr int kStepV = 128;     // K values per A stage in tensor memory (half a 256-value block)
constexpr int kAStages = 4;     // A stages: producer set J fills stages J and J + 2 in turn
constexpr int kChunkV = 64;     // K values per B chunk (one 128-byte swizzle row of f16)

// warp roles
constexpr int kTcProd = 8;                  // 0-7: A producers, two sets of four lane quadrants
constexpr int kTcMmaW = 8;                  // MMA issuer 0 (lane 0)
constexpr int kTcRawW = 9;                  // unit fetch, pair metadata, bulk copy of the quantized rows
constexpr int kTcBW = 10;                   // B tensor copies (lane 0)
constexpr int kTcEpi0 = 11;                 // 11-14: epilogue, lane quadrants 3, 0, 1, 2
constexpr int kTcMma1W = 15;                // MMA issuer 1 (lane 0), on another SM sub-partition
constexpr int kTcWarps = 16;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kMetaArrivals = 2 + 1 + 4;  // the roles that read a unit's metadata: issuers, B loader, epilogue

// tensor memory: A stages at columns [0, 256) (64 columns each), accumulators at [256, 512):
// buffer b at 256 + 128 b, split into two 64-column halves (one per issuer) for units of at
// most kSplitN tokens
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol0 = 256;
constexpr int kSplitN = 64;

// B stages of kNT rows x 128 bytes; a unit of npad tokens packs cps = 128 / npad chunks (a power
// of two) into one stage, so that small units keep as many K values in flight as large ones.
// (Measured: a fourth gate/up stage bought with a smaller codebook table, or more down stages,
// did not make the chunk faster.)
__host__ __device__ inline int tc_bstages(int MODE) { return MODE == 0 ? 3 : 6; }
__host__ __device__ inline int tc_cps(int npad, int nchunks) {
    int c = 1;
    while (2 * c * npad <= kNT && 2 * c <= nchunks) c *= 2;
    return c;
}
// a unit's K steps are shared by the two issuers (step st by issuer st & 1) when it has at most
// kSplitN tokens and at least two steps
__host__ __device__ inline bool tc_split(int npad, int nsteps) { return npad <= kSplitN && nsteps >= 2; }
// codebook as f16 pairs (exact: |value| <= 128), 8 interleaved copies (see qdot.cuh)
__device__ void build_pair_table_f16(uint4 *tab, const int8_t *__restrict__ codebook) {
    for (int e = threadIdx.x; e < 256; e += blockDim.x) {
        const uint2 raw = reinterpret_cast<const uint2 *>(codebook)[e];
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t word = p < 2 ? raw.x : raw.y;
            const int g0 = (int8_t)((word >> (16 * (p & 1))) & 0xffu);
            const int g1 = (int8_t)((word >> (16 * (p & 1) + 8)) & 0xffu);
            w[p] = (uint32_t)__half_as_ushort(__int2half_rn(g0)) | ((uint32_t)__half_as_ushort(__int2half_rn(g1)) << 16);
        }
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int c = 0; c < kTabCopies; ++c) tab[e * kTabCopies + ((c + threadIdx.x) & (kTabCopies - 1))] = v;
    }
}

// ---- unit lists ------------------------------------------------------------------------------
// A unit word: expert (bits 0-9), row tile (10-14), token block (15-31).
__host__ __device__ inline uint32_t unit_word(int e, int mt, int tb) {
    return (uint32_t)e | ((uint32_t)mt << 10) | ((uint32_t)tb << 15);
}
struct TcUnits {  // [count_gu, count_dn, next_gu, next_dn, pad..][gu units][dn units]
    uint32_t *counts, *gu, *dn;
};
__host__ __device__ inline size_t tc_max_blocks(int P, int E) { return (size_t)P / kNT + (size_t)E; }

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

// Per expert: its full 128-pair blocks first (all experts), then its partial block; each block
// times the row tiles of the mode.  Zeroes the two work counters.
__global__ void __launch_bounds__(512) tc_units_kernel(const uint32_t *__restrict__ offs, int E, int gu_tiles,
                                                       int dn_tiles, uint32_t *counts, uint32_t *gu, uint32_t *dn,
                                                       const int32_t *ctrl, int layer) {
    __shared__ uint32_t scan_s[16];
    if (ld_ctrl(ctrl) <= layer) return;
    const int e = threadIdx.x;
    const uint32_t n = e < E ? offs[e + 1] - offs[e] : 0u;
    const uint32_t full = n / kNT, part = (n % kNT) ? 1u : 0u;
    const uint2 sf = block_scan512(full, scan_s);
    const uint2 sp = block_scan512(part, scan_s);
    for (uint32_t f = 0; f < full; ++f) {
        for (int mt = 0; mt < gu_tiles; ++mt) gu[(size_t)(sf.x + f) * gu_tiles + mt] = unit_word(e, mt, (int)f);
        for (int mt = 0; mt < dn_tiles; ++mt) dn[(size_t)(sf.x + f) * dn_tiles + mt] = unit_word(e, mt, (int)f);
    }
    if (part) {
        for (int mt = 0; mt < gu_tiles; ++mt) gu[(size_t)(sf.y + sp.x) * gu_tiles + mt] = unit_word(e, mt, (int)full);
        for (int mt = 0; mt < dn_tiles; ++mt) dn[(size_t)(sf.y + sp.x) * dn_tiles + mt] = unit_word(e, mt, (int)full);
    }
    if (e == 0) {
        counts[0] = (sf.y + sp.y) * gu_tiles;
        counts[1] = (sf.y + sp.y) * dn_tiles;
        counts[2] = 0u;
        counts[3] = 0u;
    }
}

// xg[p][:] = f16(xn[pair_tok[p]][:]): the gate/up B operand in pair order, one warp per pair
__global__ void __launch_bounds__(256) tc_gather_kernel(const float *__restrict__ xn,
                                                        const uint32_t *__restrict__ pair_tok,
                                                        uint16_t *__restrict__ xg, int P, int H, const int32_t *ctrl,
                                                        int layer) {
    if (ld_ctrl(ctrl) <= layer) return;
    const int lane = threadIdx.x & 31;
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (p >= P) return;
    const float4 *src = reinterpret_cast<const float4 *>(xn + (size_t)pair_tok[p] * H);
    uint4 *dst = reinterpret_cast<uint4 *>(xg + (size_t)p * H);
    for (int c = lane; c < H / 8; c += 32) {
        const float4 a = __ldg(src + 2 * c), b = __ldg(src + 2 * c + 1);
        const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
        const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
        dst[c] = make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                            *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
    }
}

// ---- the grouped GEMM ------------------------------------------------------------------------
struct TcMeta {  // one unit, staged by the raw loader
    int end, e, mt, nvalid, npad;
    uint32_t p_lo;
    uint32_t tok[kNT];
    uint8_t kk[kNT];
};

struct TcLayout {
    size_t rawb, o_tab, o_b, o_meta, o_raw, total;
    int sb;
    __host__ __device__ TcLayout(int MODE, int H, int I) {
        sb = tc_bstages(MODE);
        rawb = align_up(MODE == 0 ? matrix_bytes(kTcRows, H) : matrix_bytes(kTcRows, I), 128);
        o_tab = 1024;
        o_b = o_tab + kTabBytes;  // 1024-aligned: the swizzle atoms
        o_meta = o_b + (size_t)sb * kNT * kChunkV * 2;
        o_raw = align_up(o_meta + 2 * sizeof(TcMeta), 128);
        total = o_raw + 2 * rawb;
    }
};

struct TcArgs {
    CUtensorMap bmap;  // B operand [P][C] f16, box 64 x 16 rows, 128-byte swizzle
    PrefillArgs a;
    TcUnits U;
};

// One 8-value group -> four f16 pairs of d * value from its table entry q (the group's
// codebook row as f16 pairs): sign bits of gs, then the scale.
__device__ __forceinline__ void group_f16(uint4 q, uint32_t gs, uint32_t dd, uint32_t *out) {
    const uint32_t s = (gs >> 8) & 0xffu;
    const uint32_t s2 = s | ((s << 15) & 0x007f0000u);  // bit 2i -> 15 and 2i+1 -> 31 after << (15 - 2i)
    const __half2 d2 = *reinterpret_cast<const __half2 *>(&dd);
    uint32_t w[4] = {q.x ^ ((s2 << 15) & 0x80008000u), q.y ^ ((s2 << 13) & 0x80008000u),
                     q.z ^ ((s2 << 11) & 0x80008000u), q.w ^ ((s2 << 9) & 0x80008000u)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&w[i]), d2);
        out[i] = *reinterpret_cast<const uint32_t *>(&v);
    }
}
// 8 groups -> 32 words, the 8 table loads issued before any arithmetic (`tabc` = shared-window
// address of this lane's copy of the table)
__device__ __forceinline__ void groups8_f16(const uint32_t (&gs)[8], uint32_t dd, uint32_t tabc, uint32_t (&out)[32]) {
    uint4 q[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) q[g] = lds128(tabc + (gs[g] & 0xffu) * (16 * kTabCopies));
#pragma unroll
    for (int g = 0; g < 8; ++g) group_f16(q[g], gs[g], dd, &out[4 * g]);
}

// Producer step: `ng` groups from flat group index G0 of the raw tile (shared-window address
// `raw`; rows of C values stored back to back in 66-byte blocks), d of block G0 >> 5.  Each
// group index is read with its own 16-bit load: a variant that loaded whole 16-byte pieces of
// the 528-byte rows and unpacked them from registers needed one unrolled copy per block and
// half and ran four times slower (instruction-cache misses).
__device__ __forceinline__ void produce_generic(uint32_t raw, int G0, int ng, uint32_t tabc, uint32_t tcol) {
    const uint32_t db = lds_u16(raw + (uint32_t)(G0 >> 5) * kBlockBytes);
    const uint32_t dd = db | (db << 16);
    for (int pc = 0; pc < ng / 8; ++pc) {
        uint32_t gs[8], out[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const int G = G0 + 8 * pc + g;
            gs[g] = lds_u16(raw + (uint32_t)(G >> 5) * kBlockBytes + 2 + 2 * (G & 31));
        }
        groups8_f16(gs, dd, tabc, out);
        tc::st32(tcol + 32 * pc, out);
    }
}

// MODE 0: gate/up -> hb (f16 h, pair order).  MODE 1: down -> outbuf (f32, (token, k) order).
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs args) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const PrefillArgs &a = args.a;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint64_t *raw_full = bars, *meta_empty = bars + 2, *a_full = bars + 4, *a_empty = bars + 8;
    uint64_t *acc_full = bars + 12, *acc_empty = bars + 14, *fin_bar = bars + 16, *meta_full = bars + 18;
    uint64_t *data_empty = bars + 20;  // the quantized rows of a buffer decoded (producers)
    uint64_t *b_full = bars + 24, *b_empty = bars + 40;  // [sb] each, sb <= 16
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(smem + 512);
    int *abort_s = reinterpret_cast<int *>(smem + 516);
    int *data_end = reinterpret_cast<int *>(smem + 520);  // [2]: no unit in this raw buffer
    const TcLayout lay(MODE, a.H, a.I);
    const int SB = lay.sb;
    uint4 *tab = reinterpret_cast<uint4 *>(smem + lay.o_tab);
    uint8_t *bst = smem + lay.o_b;  // [SB][kNT rows][128 B]
    TcMeta *meta = reinterpret_cast<TcMeta *>(smem + lay.o_meta);
    uint8_t *rawb = smem + lay.o_raw;  // [2][lay.rawb]

    if (ld_ctrl(a.ctrl) <= a.layer) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = MODE == 0 ? a.H : a.I;       // K of this GEMM (row length)
    const int nsteps = C / kStepV;               // A stages per unit (C >= 128)
    const int nchunks = C / kChunkV;             // B chunks per unit
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&meta_full[i], 1);
            mbar_init(&meta_empty[i], kMetaArrivals);
            mbar_init(&data_empty[i], kTcProd);
            mbar_init(&acc_full[i], 2);  // one arrival per issuer
            mbar_init(&acc_empty[i], 4);
        }
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&a_empty[i], 1);
        }
        mbar_init(fin_bar, 2);
        for (int i = 0; i < SB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 2);  // one arrival per issuer
        }
        *abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_s, kTmemCols);
        tc::tmem_relinquish();
    }
    build_pair_table_f16(tab, a.codebook);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_s;
    const uint32_t count = __ldcg(&args.U.counts[MODE]);
    const uint32_t *units = MODE == 0 ? args.U.gu : args.U.dn;
    bool failed = false;
    auto aborted = [&]() { return *reinterpret_cast<volatile int *>(abort_s) != 0; };
    auto fail_now = [&]() {
        if (lane == 0) atomicExch(abort_s, 1);
        failed = true;
    };
    // Bounded waits (whole warp; warp-uniform result): lane 0 polls with test_wait, which never
    // suspends.  A suspended try_wait wakes up microseconds after the phase completes, which
    // the unit-level hand-offs (metadata, accumulators) cannot afford either.
    auto wait_spin = [&](uint64_t *bar, uint32_t parity) {
        if (!mbar_spin_warp(bar, parity)) fail_now();
        return !failed;
    };
    // unit k's metadata (meta_full of its buffer: published before its quantized rows land, so
    // that the activations are requested while the weights are still on their way); NULL at the
    // end of the list or on failure
    auto next_meta = [&](uint32_t k) -> const TcMeta * {
        if (aborted() || !wait_spin(&meta_full[k & 1], (k >> 1) & 1)) return nullptr;
        const TcMeta *m = &meta[k & 1];
        return m->end ? nullptr : m;
    };

    if (warp == kTcRawW) {
        // ---------------- unit fetch + quantized rows ----------------
        // Two buffers, each released twice: its quantized rows once the producers have decoded
        // them (data_empty), its metadata once the issuers, the B loader and the epilogue are
        // done with the unit (meta_empty).  So the next rows are requested while the epilogue
        // still drains the unit before, and the metadata is published (meta_full) before the
        // rows land, so that the activations are requested in the meantime.
        // The next unit is claimed and its words, pairs and slot loaded while this one's
        // buffers are awaited: that chain of dependent loads takes a few microseconds, as long as
        // the producers take for a unit of the down GEMM.
        const size_t matb = matrix_bytes(a.I, a.H);
        struct Unit {
            bool end;
            int e, mt, nvalid;
            uint32_t p_lo, tok[kNT / 32];
            uint8_t kk[kNT / 32];
            uint64_t slot;  // lane 0
        };
        auto fetch = [&](Unit &f) {
            uint32_t u = 0;
            if (lane == 0) u = atomicAdd(&args.U.counts[2 + MODE], 1u);
            u = __shfl_sync(kFull, u, 0);
            f.end = u >= count;
            f.e = f.mt = f.nvalid = 0;
            f.p_lo = 0;
            f.slot = 0;
            if (f.end) return;
            const uint32_t uw = __ldcg(&units[u]);
            f.e = uw & 1023;
            f.mt = (uw >> 10) & 31;
            const uint32_t pe0 = __ldcg(&a.offs[f.e]), pe1 = __ldcg(&a.offs[f.e + 1]);
            f.p_lo = pe0 + (uw >> 15) * (uint32_t)kNT;
            f.nvalid = (int)min((uint32_t)kNT, pe1 - f.p_lo);
#pragma unroll
            for (int i = 0; i < kNT / 32; ++i) {
                const int n = lane + 32 * i;
                f.tok[i] = n < f.nvalid ? __ldcg(&a.pair_tok[f.p_lo + n]) : 0u;
                f.kk[i] = n < f.nvalid ? __ldcg(&a.pair_k[f.p_lo + n]) : (uint8_t)0;
            }
            if (lane == 0) f.slot = __ldcg(&a.slots[(size_t)f.tok[0] * a.K + f.kk[0]]);
        };
        uint32_t armed = 0;  // units whose raw_full phase was started (a copy or a plain arrival)
        // the quantized rows are read once per chunk: first out of L2, so that they do not push
        // out the activations, which every row tile of an expert reads again
        const uint64_t pol = l2_evict_first();
        Unit cur, nxt;
        fetch(cur);
        for (uint32_t k = 0;; ++k) {
            const int rb = k & 1;
            if (k >= 2 && (aborted() || !wait_spin(&data_empty[rb], ((k >> 1) - 1) & 1))) break;
            if (lane == 0) {
                data_end[rb] = cur.end ? 1 : 0;
                const uint64_t slot = cur.slot;
                if (cur.end) {
                    mbar_arrive(&raw_full[rb]);
                } else if (slot == 0 || (slot & 15)) {
                    // nothing is copied: the unit's outputs are garbage and the host sees the flag
                    dev_error(a.ctrl, slot == 0 ? RL_DEVERR_MISSING : RL_DEVERR_SLOT_ALIGN);
                    mbar_arrive(&raw_full[rb]);
                } else {
                    const uint8_t *rec = reinterpret_cast<const uint8_t *>(slot);
                    uint8_t *dst = rawb + rb * lay.rawb;
                    if (MODE == 0) {
                        const uint32_t b = (uint32_t)matrix_bytes(kGuUnits, a.H);
                        const uint8_t *g = rec + (size_t)cur.mt * b;
                        mbar_arrive_expect_tx(&raw_full[rb], 2 * b);
                        bulk_g2s_hint(dst, g, b, &raw_full[rb], pol);
                        bulk_g2s_hint(dst + b, g + matb, b, &raw_full[rb], pol);
                    } else {
                        const uint32_t b = (uint32_t)matrix_bytes(kTcRows, a.I);
                        mbar_arrive_expect_tx(&raw_full[rb], b);
                        bulk_g2s_hint(dst, rec + 2 * matb + (size_t)cur.mt * b, b, &raw_full[rb], pol);
                    }
                }
            }
            armed = k + 1;
            __syncwarp();
            if (!cur.end) fetch(nxt);
            if (k >= 2 && (aborted() || !wait_spin(&meta_empty[rb], ((k >> 1) - 1) & 1))) break;
            TcMeta &m = meta[rb];
#pragma unroll
            for (int i = 0; i < kNT / 32; ++i) {
                const int n = lane + 32 * i;
                if (n < cur.nvalid) {
                    m.tok[n] = cur.tok[i];
                    m.kk[n] = cur.kk[i];
                }
            }
            if (lane == 0) {
                m.end = cur.end ? 1 : 0;
                m.e = cur.e;
                m.mt = cur.mt;
                m.nvalid = cur.nvalid;
                m.npad = (cur.nvalid + 15) & ~15;
                m.p_lo = cur.p_lo;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&meta_full[rb]);
            __syncwarp();
            if (cur.end) break;
            cur = nxt;
        }
        // copies still in flight (only after a failure) must land before the CTA exits
        for (uint32_t j = armed >= 2 ? armed - 2 : 0; j < armed; ++j) mbar_wait_warp(&raw_full[j & 1], (j >> 1) & 1);
    } else if (warp == kTcBW) {
        // ---------------- B operand: tensor copies of the unit's activation rows ----------------
        uint32_t gbs = 0;  // B stages used so far
        const uint64_t pol = l2_evict_last();
        for (uint32_t k = 0;; ++k) {
            const TcMeta *m = next_meta(k);
            if (!m) break;
            const int npad = m->npad, cps = tc_cps(npad, nchunks);
            const uint32_t p_lo = m->p_lo;
            for (int bs = 0; bs < nchunks / cps; ++bs) {
                const int s = gbs % SB;
                if (gbs >= (uint32_t)SB && !wait_spin(&b_empty[s], ((gbs / SB) - 1) & 1)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&b_full[s], (uint32_t)(cps * npad * kChunkV * 2));
                    for (int j = 0; j < cps; ++j)
                        for (int r = 0; r < npad / 16; ++r)
                            tma_load_2d_hint(bst + ((size_t)s * kNT + j * npad + 16 * r) * (kChunkV * 2), &args.bmap,
                                             (bs * cps + j) * kChunkV, (int)p_lo + 16 * r, &b_full[s], pol);
                }
                __syncwarp();
                ++gbs;
            }
            if (failed) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&meta_empty[k & 1]);
        }
        // stages issued but never consumed (only after a failure) must land before the CTA exits
        for (uint32_t j = gbs >= (uint32_t)SB ? gbs - SB : 0; j < gbs; ++j) mbar_wait_warp(&b_full[j % SB], (j / SB) & 1);
    } else if (warp < kTcProd) {
        // ---------------- A producers ----------------
        // Set J decodes the unit's steps st = J, J + 2, ... (K values [128 st, 128 st + 128))
        // into stage st % 4, so it fills stages J and J + 2 in turn: one is decoded while the
        // MMAs read the other.
        const int q = warp & 3, J = warp >> 2;
        // gate/up: lanes 0-15 of a quadrant hold gate rows, 16-31 the up rows of the same hidden
        // units, so that the epilogue pairs them with one shuffle
        const int rho = MODE == 0 ? (lane < 16 ? 16 * q + lane : kGuUnits + 16 * q + lane - 16) : 32 * q + lane;
        const uint32_t tabc = smem_addr(tab + (lane & (kTabCopies - 1)));
        const uint32_t lanebase = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t used = 0u, par = 0u;  // per stage: filled before; parity of its next fill
        for (uint32_t k = 0;; ++k) {
            // the producers need the unit's rows alone, not its metadata
            if (aborted() || !wait_spin(&raw_full[k & 1], (k >> 1) & 1)) break;
            if (*reinterpret_cast<volatile int *>(&data_end[k & 1])) break;
            const uint32_t raw = smem_addr(rawb + (k & 1) * lay.rawb);
            for (int st = J; st < nsteps; st += 2) {
                const int sg = st % kAStages;
                // before fill f >= 1 of the stage, the MMAs of fill f - 1 must be done
                if (((used >> sg) & 1u) && !wait_spin(&a_empty[sg], ((par >> sg) & 1u) ^ 1u)) break;
                const uint32_t tcol = lanebase + (uint32_t)(sg * kStepV / 2);
                produce_generic(raw, rho * (C / 8) + st * (kStepV / 8), kStepV / 8, tabc, tcol);
                tc::st_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[sg]);
                used |= 1u << sg;
                par ^= 1u << sg;
            }
            if (failed) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&data_empty[k & 1]);
        }
    } else if (warp == kTcMmaW || warp == kTcMma1W) {
        // ---------------- MMA issuers: lane 0 of two warps ----------------
        // Measured on GB300: one thread issues an M = 128, K = 16 MMA at best every ~54 cycles
        // whatever N (the tensor pipe itself needs 64 cycles at N = 128), two threads issuing
        // into separate accumulators twice as many.  So a unit of at most kSplitN tokens is
        // shared: issuer I takes the K steps st with st & 1 == I (those of producer set I) into
        // its own half of the accumulator buffer; a larger unit is issued by issuer 0 alone.
        // Both issuers walk every step and every B stage of every unit, so that their stage
        // parities stay in step with the fills; a B stage or an accumulator buffer is released
        // by both (a commit where the issuer used it, a plain arrival where it did not).  The
        // issue path is kept short: descriptors built once per B chunk and advanced by
        // constants, no warp-wide synchronisation.
        if (lane == 0) {
            const int me = warp == kTcMmaW ? 0 : 1;
            auto spin1 = [&](uint64_t *bar, uint32_t parity) {
                for (uint32_t i = 0; i < kSpinPolls; ++i)
                    if (mbar_test_wait(bar, parity)) return true;
                atomicExch(abort_s, 1);
                failed = true;
                return false;
            };
            const uint32_t bst_s = tc::s_addr(bst);
            uint32_t gbs = 0, par = 0u;  // B stages passed; per A stage, parity of its next fill
            for (uint32_t k = 0; !aborted(); ++k) {
                if (!spin1(&meta_full[k & 1], (k >> 1) & 1)) break;
                const TcMeta *m = &meta[k & 1];
                if (m->end) break;
                const int npad = m->npad, cps = tc_cps(npad, nchunks);
                const bool split = tc_split(npad, nsteps);
                const uint32_t idesc = tc::instr_desc(0u, kTcRows, npad);
                const uint32_t cstride = (uint32_t)(npad * kChunkV * 2);  // bytes between the chunks of a stage
                mbar_arrive(&meta_empty[k & 1]);  // the metadata is no longer needed here
                const int ab = k & 1;
                if (k >= 2 && !spin1(&acc_empty[ab], ((k >> 1) - 1) & 1)) break;
                const uint32_t d = tmem + kAccCol0 + (uint32_t)(ab * kNT + (split ? me * kSplitN : 0));
                int s = 0, j = 0;
                uint32_t bc = 0;
                bool first = true, stage_used = false;
                for (int st = 0; st < nsteps; ++st) {
                    const int sg = st % kAStages;
                    const bool mine = split ? (st & 1) == me : me == 0;
                    if (mine) {
                        if (!spin1(&a_full[sg], (par >> sg) & 1u)) break;
                        tc::fence_after();
                    }
                    par ^= 1u << sg;
                    const uint32_t a0 = tmem + (uint32_t)(sg * kStepV / 2);
#pragma unroll
                    for (int c = 0; c < kStepV / kChunkV; ++c) {
                        if (j == 0) {
                            s = gbs % SB;
                            if (!spin1(&b_full[s], (gbs / SB) & 1)) break;
                            tc::fence_after();
                            bc = bst_s + (uint32_t)(s * kNT * kChunkV * 2);
                        }
                        if (mine) {
                            const uint64_t bd = tc::smem_desc_sw128(bc, 1024);
                            const uint32_t ac = a0 + (uint32_t)(c * kChunkV / 2);
                            if (first)
                                tc::mma_f16_ts(d, ac, bd, idesc, 0u);
                            else
                                tc::mma_f16_ts_acc(d, ac, bd, idesc);
                            tc::mma_f16_ts_acc(d, ac + 8, bd + 2, idesc);   // +32 bytes of B: start address field + 2
                            tc::mma_f16_ts_acc(d, ac + 16, bd + 4, idesc);
                            tc::mma_f16_ts_acc(d, ac + 24, bd + 6, idesc);
                            first = false;
                            stage_used = true;
                        }
                        bc += cstride;
                        if (++j == cps) {
                            if (stage_used)
                                tc::commit(&b_empty[s]);
                            else
                                mbar_arrive(&b_empty[s]);
                            stage_used = false;
                            ++gbs;
                            j = 0;
                        }
                    }
                    if (failed) break;
                    if (mine) tc::commit(&a_empty[sg]);
                }
                if (failed) break;
                if (first)
                    mbar_arrive(&acc_full[ab]);  // this issuer had no step of the unit
                else
                    tc::commit(&acc_full[ab]);
            }
        }
        __syncwarp();
    } else if (warp >= kTcEpi0) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + kAccCol0;
        for (uint32_t k = 0;; ++k) {
            const TcMeta *m = next_meta(k);
            if (!m) break;
            const int ab = k & 1;
            if (!wait_spin(&acc_full[ab], (k >> 1) & 1)) break;
            tc::fence_after();
            const int nvalid = m->nvalid, npad = m->npad, mt = m->mt;
            const bool split = tc_split(npad, nsteps);
            const uint32_t p_lo = m->p_lo;
            for (int c0 = 0; c0 < npad; c0 += 16) {
                uint32_t v[16];
                tc::ld16(trow + (uint32_t)(ab * kNT + c0), v);
                if (split) {  // the two issuers' partial sums, added in a fixed order
                    uint32_t v1[16];
                    tc::ld16(trow + (uint32_t)(ab * kNT + kSplitN + c0), v1);
                    tc::ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                }
                tc::ld_wait();
                if (MODE == 0) {
                    // lane < 16: gate row of hidden unit hu, lane + 16: its up row.  The gate lane
                    // takes columns c0..c0+7, the up lane c0+8..c0+15.
                    const bool gate = lane < 16;
                    const int hu = mt * kGuUnits + 16 * q + (lane & 15);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float mine = __uint_as_float(gate ? v[j] : v[8 + j]);
                        const float send = __uint_as_float(gate ? v[8 + j] : v[j]);
                        const float other = __shfl_xor_sync(kFull, send, 16);
                        const float g = gate ? mine : other, u = gate ? other : mine;
                        const int n = c0 + (gate ? j : 8 + j);
                        if (n < nvalid)
                            a.hb16[(size_t)(p_lo + n) * a.I + hu] = __half_as_ushort(__float2half_rn(silu(g) * u));
                    }
                } else {
                    const int orow = mt * kTcRows + 32 * q + lane;  // output row of H
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j;
                        if (n < nvalid)
                            a.outbuf[((size_t)m->tok[n] * a.K + m->kk[n]) * a.H + orow] = __uint_as_float(v[j]);
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[ab]);
                mbar_arrive(&meta_empty[k & 1]);
            }
        }
    }
    if (failed && lane == 0) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);
    // drain every tcgen05 operation this CTA issued, then release tensor memory
    __syncthreads();
    if (tid == kTcMmaW * 32 || tid == kTcMma1W * 32) tc::commit(fin_bar);  // each issuer's own MMAs
    if (tid == kTcMmaW * 32 && !mbar_wait(fin_bar, 0)) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);  // the drain did not finish
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// the B operand [rows][C] f16 as a tensor map: boxes of 64 values x 16 rows, 128-byte swizzle
static rl_status b_tensor_map(CUtensorMap *map, const uint16_t *base, int rows, int C) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (!enc) return fail(RL_ERR_CUDA, "moe_prefill_chunk: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t gdim[2] = {(cuuint64_t)C, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kChunkV, 16u};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult cr = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(base), gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(RL_ERR_CUDA, "moe_prefill_chunk: tensor map rejected (error %d)", (int)cr);
    return RL_OK;
}

template <int MODE>
static rl_status launch_tc(const TcArgs &args, int grid, cudaStream_t s) {
    const TcLayout lay(MODE, args.a.H, args.a.I);
    auto kern = tc_gemm_kernel<MODE>;
    rl_status st = allow_smem((const void *)kern, lay.total);
    if (st != RL_OK) return st;
    kern<<<grid, kTcThreads, lay.total, s>>>(args);
    return check_launch(MODE == 0 ? "moe_prefill_chunk gate/up" : "moe_prefill_chunk down");
}

static rl_status run_tc(const PrefillArgs &a, cudaStream_t s) {
    const int P = a.P, E = a.E;
    const int gu_tiles = a.I / kGuUnits, dn_tiles = a.H / kTcRows;
    TcUnits U;
    uint8_t *ub = reinterpret_cast<uint8_t *>(a.units);
    U.counts = reinterpret_cast<uint32_t *>(ub);
    const size_t nb = tc_max_blocks(P, E);
    U.gu = reinterpret_cast<uint32_t *>(ub + 256);
    U.dn = U.gu + nb * gu_tiles;
    tc_gather_kernel<<<(P + 7) / 8, 256, 0, s>>>(a.xn, a.pair_tok, a.xb16, P, a.H, a.ctrl, a.layer);
    tc_units_kernel<<<1, 512, 0, s>>>(a.offs, E, gu_tiles, dn_tiles, U.counts, U.gu, U.dn, a.ctrl, a.layer);
    rl_status st = check_launch("moe_prefill_chunk setup");
    if (st != RL_OK) return st;
    const int sms = sm_count();
    TcArgs args;
    args.a = a;
    args.U = U;
    const int P16 = P > 16 ? P : 16;  // rows of the operand buffers (the workspace holds at least 16)
    st = b_tensor_map(&args.bmap, a.xb16, P16, a.H);
    if (st != RL_OK) return st;
    const int g_gu = (int)std::min<size_t>(sms, nb * gu_tiles), g_dn = (int)std::min<size_t>(sms, nb * dn_tiles);
    st = launch_tc<0>(args, g_gu, s);
    if (st != RL_OK) return st;
    st = b_tensor_map(&args.bmap, a.hb16, P16, a.I);
    if (st != RL_OK) return st;
    st = launch_tc<1>(args, g_dn, s);
    if (st != RL_OK) return st;
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
    return run_tc(a, as_stream(stream));
}
