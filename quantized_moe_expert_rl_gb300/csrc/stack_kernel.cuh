// stack_kernel.cuh - the fused decode stack: ONE persistent kernel runs a run of layers of one token,
//   x <- x + sum_{k in order} w_k * down_k(silu(gate_k xn) * (up_k xn)),  xn = RMSNorm(x),
// with the router, the selection, the residency lookup, the miss count and the early-out flag
// of every layer inside the same launch.
//
// Red Lite dev38 - decode lanes, "Finding": on the pages' GPU the serialization between the
// many small decode kernels, not the bandwidth of any one of them, was the dominant waste.
// Red Lite dev21 - GPU-routed decode, "What changed": no host round trip sits between the
// router and the experts.  Red Lite dev23 - per-layer early-out, "What changed" item 1: the
// layer that selects a non-resident expert raises the flag and nothing after it runs.
//
// Design: one CTA per SM (cooperative launch, so all CTAs are co-resident), 16 warps each.
// Every CTA owns a fixed slice of each phase's work for the whole launch:
//   gate/up (expert, row) pairs [p0, p1); down output rows [q0, q0+nq), i.e. its slice of x.
// The router is split by columns, not rows: CTA b holds columns [q0, q0+nq) of every router row
// in shared memory (copied a layer ahead; they do not depend on x) and, as soon as its slice of
// x_l is final, adds its partial dot of every row into the layer's logit accumulators.  The
// accumulators are 64-bit fixed point (2^-36 resolution), so the sum is exact up to the
// rounding of each f32 partial and does not depend on the order in which the CTAs arrive.  With
// rs the RMSNorm scale, logit_e = rs * sum_h W[e][h] x[h] + bias_e, the same linear map as
// W (rs x).  This takes the router off the critical path: no barrier separates x_l from the
// selection other than the one that publishes x_l itself.
// Per launch: CTA 0 clears the accumulators, grid barrier, every CTA adds its dots on x_layer0,
// grid barrier.  Per layer:
//   B  x_l (L2) -> RMSNorm scale; logits from the accumulators; every CTA selects the top-k
//      itself (the same code on the same data gives the same ids everywhere, so no further
//      exchange is needed); CTA 0 writes the outputs, the miss count and the flag; a miss (or
//      the flag) stops every CTA.  Then the CTA's gate/up rows of the K selected experts are
//      copied into shared memory with bulk asynchronous copies;
//   C  gate/up + SwiGLU of the CTA's pairs -> h (L2); then the last warp copies the CTA's down
//      rows of the K experts and the next layer's router columns;  grid barrier
//   D  the renormalised weights (one warp); the CTA's rows of every expert's down projection,
//      the ordered combine and the residual -> its slice of x_{l+1} (L2), then its router dots
//      of layer l+1 on that slice;  grid barrier.
// Only the copies C needs first sit between the selection and the gate/up compute.
// The arithmetic of every expert row, of the RMSNorm scale and of the selection is the one the
// per-layer kernels (rl_route, moe_decode) use; the logits differ from rl_route's only by the
// order of summation (rl_route: one f32 dot per row).
//
// Grid barrier: a 64-bit arrival counter in the workspace that only ever grows (release
// reduction to arrive, acquire loads to poll).  The first arrival of a launch rounds its value
// down to a multiple of the grid size to find the base, so no reset is needed between launches.  Every spin is bounded: on expiry the CTA sets
// RL_DEVERR_WAIT_TIMEOUT, waits (bounded) for its own copies in flight and returns; the other
// CTAs then time out at their next barrier.
#pragma once
#include <map>
#include <mutex>
#include <tuple>

#include "decode_rows.cuh"
#include "select.cuh"

namespace rl {

constexpr int kStThreads = 512;
constexpr int kStWarps = kStThreads / 32;
constexpr int kStGuChunks = 2;
constexpr int kStBars = 3 + 2 * kStGuChunks;  // [0] down rows, [1] router columns, [2..] gate/up chunks, [last] table row
constexpr uint32_t kSpinCap = 1u << 22;       // global-memory polls (~1 us each): seconds
// Test knobs in the workspace header (zero = off), so that a test can make the bounded waits
// run out without faulting anything: the u32 at byte 64 replaces every wait limit of the
// launch (polls of the grid barrier, of the copy barriers); the i32 at byte 68, when n > 0,
// makes CTA n - 1 leave before its first grid-barrier arrival (the other CTAs' waits at that
// barrier run out) and, when n < 0, makes CTA -n - 1 expect 16 bytes more than its first
// router-column copy brings (its own wait on that copy runs out, the others then wait in vain
// at the next grid barrier).
constexpr int kStKnobWord = 16;  // u32 index of the knobs in the workspace header
constexpr int kStHdr = 1024;                  // barriers, scalars, CTA constants, outputs of the selection
constexpr int kStPredMax = 32;                // experts prefetched on the pre-gated prediction
constexpr int kStCand = 16;                   // single-warp selection: candidates per lane (E <= 512)
// selection scratch: the producer warp's 32 lane maxima, 32 (key, id) candidates and kMaxK
// results, the layer's 512 keys, then its residency row (u64, copied ahead)
constexpr int kStSelKeys = 128 + 256 + 4 * kMaxK;  // then the 512 keys of the layer
constexpr int kStSelTab = kStSelKeys + 512 * 4;
constexpr int kStSelBytes = kStSelTab + 512 * 8;
static_assert(kStSelTab % 16 == 0, "the residency row copy needs a 16-byte aligned destination");
// The warp that issues every bulk copy.  A memory fence waits for the bulk copies its own
// thread has in flight, so the thread that runs the grid barrier (thread 0) never issues one.
constexpr int kStProducer = kStWarps - 1;
// Router partial sums in 64-bit fixed point, value * 2^36 rounded to an integer: a partial is
// limited to |p| < 2^19, so the sum of up to 2^8 of them (one per CTA) stays inside int64.
constexpr float kFixScale = 68719476736.0f;         // 2^36
constexpr float kFixInv = 1.4551915228366852e-11f;  // 2^-36
constexpr float kFixMax = 524288.0f;                // 2^19
constexpr int kStMaxGrid = 256;

// down rows handled together so that every copy starts on a block boundary (rows * I % 2048 == 0)
__host__ __device__ inline int dn_unit(int I) { return I >= 2048 ? 1 : 2048 / I; }
// a CTA's slice of x (its down rows) is made of whole down units and of whole 8-float groups,
// so that its router columns are whole 32-byte DRAM sectors; CTA b owns rows [b dmax, b dmax +
// dmax) (fewer for the last, none past H), so every busy CTA takes the same column box
__host__ __device__ inline int dq_unit(int I) { return dn_unit(I) > 8 ? dn_unit(I) : 8; }
// router rows per column box (a tensor copy moves at most 256 rows) and boxes per layer
__host__ __device__ inline int rc_nbox(int E) { return (E + 255) / 256; }
__host__ __device__ inline int rc_rows(int E) { return (E + rc_nbox(E) - 1) / rc_nbox(E); }

struct StLayout {
    int rmax, dmax, rowb, dtileb;
    size_t rbs, rcb, o_xt, o_rc, o_xq, o_part, o_gu, o_dn, o_o, o_h, o_sel, total;
    __host__ __device__ StLayout(int H, int E, int K, int I, int G, bool pg) {
        const int U = gu_unit(H), units = K * I / U;
        rmax = ((units + G - 1) / G) * U;
        const int Ud = dq_unit(I), gq = H / Ud;
        dmax = ((gq + G - 1) / G) * Ud;
        rbs = align_up((size_t)rc_rows(E) * dmax * sizeof(float), 128);  // one column box, 128-byte aligned
        rcb = (size_t)rc_nbox(E) * rbs;
        rowb = (int)matrix_bytes(1, H);
        dtileb = (int)align_up(matrix_bytes(dmax, I), 16);
        o_xt = kStHdr + kTabBytes;                               // x, lane-transposed for the gate/up lanes
        o_rc = align_up(o_xt + (size_t)H * sizeof(float), 128);
        // router columns [q0, q0 + dmax) of every row of one layer (and of the next, pre-gating)
        o_xq = o_rc + (pg ? 2 : 1) * rcb;
        o_part = o_xq + align_up((size_t)dmax * sizeof(float), 16);  // this CTA's slice of x
        o_gu = o_part + align_up((size_t)rmax * 4 * sizeof(float), 16);
        o_dn = o_gu + 2 * (size_t)rmax * rowb;
        o_o = o_dn + (size_t)K * dtileb;
        o_h = o_o + align_up((size_t)K * dmax * sizeof(float), 16);
        o_sel = o_h + (size_t)K * I * sizeof(float);  // h of every expert, staged for the down rows
        total = o_sel + kStSelBytes;                     // selection scratch
    }
};

// This CTA's fixed share of every phase and its shared-memory layout, kept in shared memory
// (read where needed) so that the layer loop keeps few registers live.
struct StCta {
    int p0, p1, ka, kb, n0, n1;  // gate/up (expert, row) pairs: two segments (experts ka, kb)
    int q0, nq;                  // down output rows = this CTA's slice of x
    int rowb, dtileb, dmax, rbs, rcb;
    uint32_t o_xt, o_rc, o_xq, o_part, o_gu, o_dn, o_o, o_h, o_sel;
};

struct StackArgs {
    CUtensorMap wmap;        // the router weights as a [L * E][H] f32 matrix; box rc_rows x dmax
    float *x;
    float eps;
    const float *W;          // [L][E][H]
    const float *bias;       // [L][E] or NULL
    const uint64_t *table;   // [L][E]
    const int8_t *codebook;  // [256][8]
    int32_t *ids;            // [L][K]
    float *weights;          // [L][K]
    uint64_t *slots;         // [L][K]
    uint32_t *miss;          // [L]
    int32_t *ctrl;
    float *logits_out;  // [L][E] or NULL
    float *x_hist;      // [L][H] or NULL
    unsigned long long *ctr;
    long long *acc;     // [2][E] fixed-point router sums, by layer parity
    long long *acc_pg;  // [2][E] the same for the pre-gate dots (next layer's router, this input)
    long long *ss;      // [2] sums of squares of x (rms_scale_warp's fixed point), by layer parity
    float *h;           // [K][I]
    uint32_t *pg_hits;  // [L] or NULL
    uint64_t *table_w;         // the table again, written by device fills (NULL without fill tables)
    const uint64_t *fill_src;  // [L][E] device-readable record sources, or NULL (stop on a miss instead)
    const uint64_t *fill_dst;  // [L][E] HBM slots
    uint32_t *filled;          // experts filled by the device
    float *y;                  // one layer without residual: y = MoE(xn), x left unchanged (NULL: the stack)
    int layer0, nl, H, E, K, I, pregate, n_layers;
};


__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// *dst += p * 2^36 rounded to an integer (a reduction performed in L2).  Integer addition is
// associative, so the sum does not depend on the order in which the CTAs arrive.
__device__ __forceinline__ void red_fixed(long long *dst, float p, int32_t *ctrl) {
    if (!(fabsf(p) < kFixMax)) {
        dev_error(ctrl, RL_DEVERR_RANGE);
        p = 0.f;
    }
    atomicAdd(reinterpret_cast<unsigned long long *>(dst), (unsigned long long)float_to_ll(p * kFixScale));
}
__device__ __forceinline__ float fixed_value(long long v) { return ll_to_float(v) * kFixInv; }

// All CTAs of the grid meet; writes before it (through L2) are visible after it.  Thread 0
// keeps the barrier target in a register; `target` = 0 means "not yet based".  The arrival is a
// release at GPU scope and the poll an acquire: together with the CTA barriers on both sides
// they order every thread's writes before the meeting against every thread's reads after it.
// Only the first arrival of a launch needs the counter's old value (to find the base); the
// later ones are reductions that thread 0 does not wait for.
__device__ __forceinline__ bool grid_sync(unsigned long long *ctr, unsigned long long &target, int *ok_s,
                                          int32_t *ctrl, uint32_t cap) {
    cta_sync();
    if (threadIdx.x == 0) {
        if (target == 0ull) {
            unsigned long long old;
            asm volatile("atom.add.release.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(ctr) : "memory");
            target = old - old % gridDim.x + 1ull;  // +1 marks "based"
        } else {
            asm volatile("red.add.release.gpu.global.u64 [%0], 1;" ::"l"(ctr) : "memory");
        }
        target += gridDim.x;
        bool ok = false;
        for (uint32_t i = 0; i < cap; ++i)
            if (ld_acquire_u64(ctr) >= target - 1ull) {
                ok = true;
                break;
            }
        if (!ok) dev_error(ctrl, RL_DEVERR_WAIT_TIMEOUT);
        *ok_s = ok;
    }
    cta_sync();  // also rejoins warp 0 after thread 0's wait
    return *ok_s != 0;
}

// chunk c of gate/up segment `seg` holds rows [cut, cut') of the segment
__device__ __forceinline__ int gu_cut(const StCta &c, int U, int seg, int ch) {
    return ((seg == 0 ? c.n0 : c.n1) / U * ch / kStGuChunks) * U;
}

// NV = H / 128 float4 columns per lane of x; GPL, SPLIT: gate/up lane geometry (moe_decode);
// DGPL, LPR: down lane geometry; FILL: the variant with device fills (moe_decode_stack_fill),
// compiled apart so that the common variant carries none of its code.
template <int NV, int GPL, int SPLIT, int DGPL, int LPR, bool FILL>
__global__ void __launch_bounds__(kStThreads, 1) stack_kernel(const __grid_constant__ StackArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint64_t *bar_dn = bars, *bar_rc = bars + 1, *bar_gu = bars + 2, *bar_tab = bars + 2 + 2 * kStGuChunks;
    float *scale_s = reinterpret_cast<float *>(smem + 64);
    int *stop_s = reinterpret_cast<int *>(smem + 68);
    int *ok_s = reinterpret_cast<int *>(smem + 72);
    int *iss_s = reinterpret_cast<int *>(smem + 76);  // copies issued at the end of C: bit 0 down rows, bit 1 router columns, bit 2 residency row
    uint32_t *cap_s = reinterpret_cast<uint32_t *>(smem + 80);  // wait limits: grid barrier, copy spin, copy wait
    int *hold_s = reinterpret_cast<int *>(smem + 92);           // test knob (see kStKnobWord)
    StCta &C = *reinterpret_cast<StCta *>(smem + 128);
    uint64_t *slots_s = reinterpret_cast<uint64_t *>(smem + 256);
    float *w_s = reinterpret_cast<float *>(smem + 384);   // [K] weights
    float *sv_s = reinterpret_cast<float *>(smem + 448);  // [K] selected logits (weights computed in D)
    int *pred_s = reinterpret_cast<int *>(smem + 512);  // [kStPredMax] predicted ids of the next layer
    int *fid_s = reinterpret_cast<int *>(smem + 640);    // [K] selected ids, for a device fill
    uint32_t *fmask_s = reinterpret_cast<uint32_t *>(smem + 704);  // selections k to fill on the device
    uint4 *tab = reinterpret_cast<uint4 *>(smem + kStHdr);
    constexpr int H = NV * 128;
    constexpr int U = H >= 2048 ? 1 : 2048 / H;  // gu_unit(H)
    static_assert(2 * DGPL <= LPR, "the h staging swizzle sl ^ q needs q < LPR");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool pregate = a.pregate > 0;

    if (threadIdx.x == 0) {
        const int E = a.E, K = a.K, I = a.I, G = gridDim.x, b = blockIdx.x;
        const StLayout lay(H, E, K, I, G, pregate);
        const int units = K * I / U;
        C.p0 = (int)((long long)b * units / G) * U;
        C.p1 = (int)((long long)(b + 1) * units / G) * U;
        const bool has = C.p1 > C.p0;
        C.ka = has ? C.p0 / I : 0;
        C.kb = has ? (C.p1 - 1) / I : 0;
        C.n0 = has ? (C.ka == C.kb ? C.p1 : (C.ka + 1) * I) - C.p0 : 0;
        C.n1 = (C.p1 - C.p0) - C.n0;
        C.q0 = b * lay.dmax < H ? b * lay.dmax : H;
        C.nq = H - C.q0 < lay.dmax ? H - C.q0 : lay.dmax;
        C.rowb = lay.rowb;
        C.dtileb = lay.dtileb;
        C.dmax = lay.dmax;
        C.rbs = (int)lay.rbs;
        C.rcb = (int)lay.rcb;
        C.o_xt = (uint32_t)lay.o_xt; C.o_rc = (uint32_t)lay.o_rc; C.o_xq = (uint32_t)lay.o_xq;
        C.o_part = (uint32_t)lay.o_part; C.o_gu = (uint32_t)lay.o_gu; C.o_dn = (uint32_t)lay.o_dn;
        C.o_o = (uint32_t)lay.o_o; C.o_h = (uint32_t)lay.o_h; C.o_sel = (uint32_t)lay.o_sel;
        for (int i = 0; i < kStBars; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *iss_s = 0;
        const uint32_t *knob = reinterpret_cast<const uint32_t *>(a.ctr) + kStKnobWord;
        const uint32_t cap = __ldcg(knob);
        cap_s[0] = cap ? cap : kSpinCap;
        cap_s[1] = cap ? cap : kSpinPolls;
        cap_s[2] = cap ? cap : kWaitCap;
        *hold_s = (int)__ldcg(knob + 1);
    }
    build_pair_table(tab, a.codebook, nullptr);  // ends with __syncthreads
    const int flag0 = ld_ctrl(a.ctrl);
    if (flag0 < a.layer0) return;  // an earlier layer already stopped the chain

    const int E = a.E;
    const int me = threadIdx.x;  // the router row (expert) whose columns this thread handles
    const uint32_t cap_grid = cap_s[0], cap_spin = cap_s[1], cap_wait = cap_s[2];
    const int hold = *hold_s;
    constexpr int kColThread = kStProducer * 32 + 31;  // issues the router column copies
    // Router columns [q0, q0 + dmax) of every row of layer index i (and of layer index i + 1
    // for the pre-gate dots) into shared memory: tensor copies of rc_rows(E) x dmax floats
    // (columns past H read as zeros), completion on bar_rc, whose n-th phase is layer index n.
    // They depend on nothing computed, so they are requested a layer ahead.
    auto issue_cols = [&](int i) {
        const int nb = (pregate && i + 1 < a.nl) ? 2 : 1, nbox = rc_nbox(E), rows = rc_rows(E);
        const uint32_t extra = (i == 0 && hold == -(int)blockIdx.x - 1) ? 16u : 0u;  // test knob
        mbar_arrive_expect_tx(bar_rc, (uint32_t)(nb * C.rcb) + extra);
        for (int q = 0; q < nb; ++q)
            for (int k = 0; k < nbox; ++k)
                tma_load_2d(smem + C.o_rc + (size_t)q * C.rcb + (size_t)k * C.rbs, &a.wmap,
                            C.q0, (a.layer0 + i + q) * E + k * rows, bar_rc);
    };
    // The residency row of layer index i into shared memory (read by every warp's selection);
    // completion on bar_tab, whose n-th phase is layer index n.  Rows are 16-byte pieces when E
    // is even; otherwise the selection reads the table through L2.
    const bool tab_smem = (E & 1) == 0 && (reinterpret_cast<uintptr_t>(a.table) & 15) == 0;
    const uint64_t *table_s = reinterpret_cast<const uint64_t *>(smem + C.o_sel + kStSelTab);
    auto issue_tab = [&](int i) {
        mbar_arrive_expect_tx(bar_tab, (uint32_t)(E * sizeof(uint64_t)));
        bulk_g2s(smem + C.o_sel + kStSelTab, a.table + (size_t)(a.layer0 + i) * E, (uint32_t)(E * sizeof(uint64_t)), bar_tab);
    };
    // The gate/up copies of the CTA's row pairs (the producer warp, whole warp): lane i <
    // 2 * kStGuChunks issues chunk (segment i / kStGuChunks, part i % kStGuChunks), its gate
    // rows and its up rows, completion on bar_gu[i]; sa, sb: the records of experts ka and kb.
    // Only the copies C needs first are issued here; the down rows and the next layer's router
    // columns wait until the end of C.
    auto issue_gu = [&](uint64_t sa, uint64_t sb) {
        fence_proxy_async_smem();
        if (FILL) asm volatile("fence.proxy.async.global;" ::: "memory");  // records filled by the device
        const int I = a.I, rowb = C.rowb;
        const size_t matb = matrix_bytes(I, H);
        if (lane < 2 * kStGuChunks && C.p1 > C.p0) {
            const int seg = lane / kStGuChunks, ch = lane % kStGuChunks;
            const int n = seg == 0 ? C.n0 : C.n1;
            const int r0 = gu_cut(C, U, seg, ch), r1 = gu_cut(C, U, seg, ch + 1);
            if (r1 > r0) {
                const uint8_t *base = reinterpret_cast<const uint8_t *>(seg == 0 ? sa : sb);
                const int ia = seg == 0 ? C.p0 - C.ka * I : 0;
                const uint32_t bytes = (uint32_t)((r1 - r0) * rowb);
                uint8_t *gdst = smem + C.o_gu + (seg == 0 ? 0 : 2 * (size_t)C.n0 * rowb) + (size_t)r0 * rowb;
                mbar_arrive_expect_tx(&bar_gu[lane], 2 * bytes);
                bulk_g2s(gdst, base + (size_t)(ia + r0) * rowb, bytes, &bar_gu[lane]);
                bulk_g2s(gdst + (size_t)n * rowb, base + matb + (size_t)(ia + r0) * rowb, bytes, &bar_gu[lane]);
            }
        }
        if (lane == 0) *iss_s = 0;
        __syncwarp();
    };
    // This CTA's partial router dots of layer index i on its slice of x_{layer0 + i} (in the
    // shared xq slice), added into acc[i & 1]; pre-gating, the next layer's dots into
    // acc_pg[i & 1].  The columns have landed (bar_rc, waited by the caller).  Each dot runs
    // over the float4 chunks of its row starting at chunk (me / 2) mod (nq / 4): rows are 16 *
    // nq bytes apart, so 8 consecutive rows read in step would share banks; the rotation (a
    // fixed order per row) spreads them.
    auto add_partials = [&](int i) {
        const int nq = C.nq;
        if (warp * 32 < nq) {
            // the sum of squares of the slice, in rms_scale_warp's groups of 8 (the slice starts
            // on a multiple of 8): one fixed-point partial per warp into ss[i & 1]
            const float *xs = reinterpret_cast<const float *>(smem + C.o_xq);
            const int t = threadIdx.x;
            const float sg = sq8_lanes(t < nq ? xs[t] : 0.f);
            bool rg = false;
            long long v = ((t & 7) == 0 && t < nq) ? sq_fixed(sg, rg) : 0ll;
            v = warp_sum_ll(v);
            if (__any_sync(kFull, rg) && lane == 0) dev_error(a.ctrl, RL_DEVERR_RANGE);
            if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long *>(a.ss + (i & 1)), (unsigned long long)v);
        }
        if (me < E && nq > 0) {
            const float4 *xq = reinterpret_cast<const float4 *>(smem + C.o_xq);
            const int rows = rc_rows(E);
            const float4 *wr = reinterpret_cast<const float4 *>(smem + C.o_rc + (size_t)(me / rows) * C.rbs) +
                               (size_t)(me % rows) * (C.dmax / 4);
            const int n4 = nq / 4, rot = (me >> 1) % n4;
            float p = 0.f;
            for (int j = 0; j < n4; ++j) {
                const int c = j + rot < n4 ? j + rot : j + rot - n4;
                const float4 w = wr[c], v = xq[c];
                p = fmaf(w.x, v.x, p); p = fmaf(w.y, v.y, p); p = fmaf(w.z, v.z, p); p = fmaf(w.w, v.w, p);
            }
            red_fixed(a.acc + (size_t)(i & 1) * E + me, p, a.ctrl);
            if (pregate && i + 1 < a.nl) {
                wr += C.rcb / sizeof(float4);
                float q = 0.f;
                for (int j = 0; j < n4; ++j) {
                    const int c = j + rot < n4 ? j + rot : j + rot - n4;
                    const float4 w = wr[c], v = xq[c];
                    q = fmaf(w.x, v.x, q); q = fmaf(w.y, v.y, q); q = fmaf(w.z, v.z, q); q = fmaf(w.w, v.w, q);
                }
                red_fixed(a.acc_pg + (size_t)(i & 1) * E + me, q, a.ctrl);
            }
        }
    };

    unsigned long long target = 0;  // grid barrier state (thread 0)
    bool ex_issued = false;         // this layer's expert copies are in flight
    int rc_pend = -1;               // layer index whose router columns are in flight (-1: none)
    bool failed = false;
    int tab_pend = -1;              // layer index whose residency row copy is in flight (-1: none)
    // ---- prologue: the accumulators start from zero (CTA 0 clears them; a grid barrier orders
    // the clear before any CTA's sums), then every CTA adds the dots of its slice of x_{layer0}
    if (C.nq > 0) {
        if (threadIdx.x == kColThread) issue_cols(0);
        rc_pend = 0;
    }
    if (tab_smem) {
        if (threadIdx.x == kColThread) issue_tab(0);
        tab_pend = 0;
    }
    if (blockIdx.x == 0) {
        for (int j = threadIdx.x; j < 2 * E; j += kStThreads) {
            __stcg(a.acc + j, 0ll);
            __stcg(a.acc_pg + j, 0ll);
        }
        if (threadIdx.x < 2) __stcg(a.ss + threadIdx.x, 0ll);
    }
    if ((int)threadIdx.x < C.nq) reinterpret_cast<float *>(smem + C.o_xq)[threadIdx.x] = __ldcg(a.x + C.q0 + threadIdx.x);
    if (hold == (int)blockIdx.x + 1) failed = true;  // test knob: this CTA never arrives
    if (!failed && !grid_sync(a.ctr, target, ok_s, a.ctrl, cap_grid)) failed = true;
    if (!failed) {
        if (warp == 0 && C.nq > 0 && !mbar_spin_warp(bar_rc, 0u, cap_spin)) failed = true;
        failed = cta_sync_or(failed) != 0;
    }
    if (!failed) {
        rc_pend = -1;
        add_partials(0);
        if (!grid_sync(a.ctr, target, ok_s, a.ctrl, cap_grid)) failed = true;
    }
    uint32_t ph = 0;
    for (int i = 0; !failed && i < a.nl; ++i, ph ^= 1u) {
        const int l = a.layer0 + i;
        const bool last = i + 1 == a.nl;
        ex_issued = false;
        // ---------------- B: the logits and the selection (the producer warp), x_l ----------------
        // Every thread reads its expert's logit accumulator (coalesced), the layer's sum of
        // squares and its share of x_l, forms its key and writes it to shared memory; after one
        // CTA barrier the producer warp selects the top-k from the keys, looks the experts up,
        // issues the expert copies, then records the selection and (CTA 0) writes the outputs,
        // the miss count and the flag.  The other warps stage x_l for the gate/up lanes
        // meanwhile; a second CTA barrier ends the phase.
        constexpr int kXv = (H / 4 + kStThreads - 1) / kStThreads;
        float4 xv_r[kXv];  // this thread's share of x_l, staged below
        const long long accv = me < E ? __ldcg(a.acc + (size_t)(i & 1) * E + me) : 0ll;
        const float biasv = (a.bias && me < E) ? __ldcg(a.bias + (size_t)l * E + me) : 0.f;
        const long long ssv = __ldcg(a.ss + (i & 1));
#pragma unroll
        for (int u = 0; u < kXv; ++u) {
            const int j = threadIdx.x + u * kStThreads;
            xv_r[u] = j < H / 4 ? __ldcg(reinterpret_cast<const float4 *>(a.x) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // acc_pg[(i + 1) & 1] was last read in D of the previous layer; it takes this
        // layer's pre-gate sums next
        if (pregate && i > 0 && blockIdx.x == 0)
            for (int j = threadIdx.x; j < E; j += kStThreads) __stcg(a.acc_pg + (size_t)((i + 1) & 1) * E + j, 0ll);
        uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem + C.o_sel + kStSelKeys);
        {
            // logit = rs * (W x) + bias: the RMSNorm scale applied to the summed dots
            const float rs = a.eps >= 0.f ? rms_scale_from(ssv, H, a.eps) : 1.f;
            uint32_t key = 0u;
            if (me < E) {
                const float lv = fmaf(fixed_value(accv), rs, biasv);
                key = order_key(lv);
                if (blockIdx.x == 0) {
                    if (lv != lv) dev_error(a.ctrl, RL_DEVERR_NAN);
                    if (a.logits_out) a.logits_out[(size_t)l * E + me] = lv;
                }
            }
            keys_s[me] = key;
            if (threadIdx.x == 0) *scale_s = rs;
        }
        cta_sync();
        bool early = false;  // the producer warp issued the gate/up copies from its own selection
        if (warp == kStProducer) {
            const int K = a.K;
            uint32_t kk[16];  // in sel_id's layout: conflict-free 8-byte reads
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint2 v = reinterpret_cast<const uint2 *>(keys_s)[32 * c + lane];
                kk[2 * c] = v.x;
                kk[2 * c + 1] = v.y;
            }
            int my_id;
            float my_val;
            {
                uint8_t *ws = smem + C.o_sel;
                warp_topk_thr(kk, E, K, reinterpret_cast<uint32_t *>(ws), reinterpret_cast<uint2 *>(ws + 128),
                              reinterpret_cast<int *>(ws + 384), my_id, my_val);
            }
            uint64_t slot = 0;
            if (tab_smem) {
                if (!mbar_spin_warp(bar_tab, (uint32_t)(i & 1), cap_spin)) failed = true;
                if (lane < K) slot = table_s[my_id];
            } else if (lane < K) {
                slot = __ldcg(a.table + (size_t)l * E + my_id);
            }
            __syncwarp();
            // the decisions of every CTA follow from the same selection
            const unsigned mmask = __ballot_sync(kFull, lane < K && slot == 0);
            const int nmiss = __popc(mmask);
            const bool bad = __ballot_sync(kFull, lane < K && slot != 0 && (slot & 15)) != 0;
            // with fill tables, a miss whose record has a source is filled here by the device
            // instead of stopping the launch
            bool fillable = FILL && nmiss > 0;
            if (FILL && fillable) {
                const size_t at = (size_t)l * a.E + (lane < K ? my_id : 0);
                const bool ok = !(lane < K && slot == 0) ||
                                (a.fill_src[at] != 0 && a.fill_dst[at] != 0 && ((a.fill_src[at] | a.fill_dst[at]) & 15) == 0);
                fillable = __all_sync(kFull, ok);
            }
            const bool stop = (nmiss > 0 && !fillable) || bad || flag0 <= l || failed;
            if (!stop && !(FILL && nmiss > 0)) {
                issue_gu(__shfl_sync(kFull, slot, C.ka), __shfl_sync(kFull, slot, C.kb));
                early = true;
            }
            {
                if (lane < K) {
                    slots_s[lane] = slot;
                    sv_s[lane] = my_val;
                    fid_s[lane] = my_id;
                }
                if (FILL && lane == 0) *fmask_s = fillable && !stop ? mmask : 0u;
                __syncwarp();
                if (blockIdx.x == 0 && a.pg_hits && pregate && i > 0) {
                    // how many of this layer's experts the previous layer predicted
                    bool hit = false;
                    for (int j = 0; j < a.pregate; ++j) hit |= lane < K && pred_s[j] == my_id;
                    const int nhit = __popc(__ballot_sync(kFull, hit));
                    if (lane == 0) a.pg_hits[l] = (uint32_t)nhit;
                }
                if (blockIdx.x == 0) {
                    if (lane < K) {
                        a.ids[(size_t)l * K + lane] = my_id;
                        a.slots[(size_t)l * K + lane] = slot;
                    }
                    if (stop) {  // the caller resumes from this layer's outputs: its weights now
                        const float w = topk_weight(my_val, K);
                        if (lane < K) a.weights[(size_t)l * K + lane] = w;
                    }
                    if (lane == 0 && nmiss > 0) {
                        atomicAdd(a.miss + l, (uint32_t)nmiss);
                        if (!fillable) atomicMin(a.ctrl, l);
                    }
                    if (lane == 0 && bad) dev_error(a.ctrl, RL_DEVERR_SLOT_ALIGN);
                }
                if (lane == 0) *stop_s = stop;
            }
        }
        {
            // x_l lane-transposed for the gate/up lanes: float4 q of the slice of lane L of row
            // half h (columns h H/SPLIT + L 8 GPL ...) sits at [h][q][L ^ q] (the xor spreads
            // the staging writes of consecutive q over the banks)
            float4 *xt_s = reinterpret_cast<float4 *>(smem + C.o_xt);
#pragma unroll
            for (int u = 0; u < kXv; ++u) {
                const int j = threadIdx.x + u * kStThreads;
                if (j >= H / 4) break;
                const int hf = H / 4 / SPLIT, h = j / hf, r = j % hf, L = r / (2 * GPL), q = r % (2 * GPL);
                xt_s[(h * 2 * GPL + q) * 32 + (L ^ q)] = xv_r[u];
            }
        }
        if (a.x_hist && blockIdx.x == 0)
            for (int j = threadIdx.x; j < H / 4; j += kStThreads)
                reinterpret_cast<float4 *>(a.x_hist + (size_t)l * H)[j] = __ldcg(reinterpret_cast<const float4 *>(a.x) + j);
        tab_pend = -1;
        cta_sync();
        if (*stop_s) break;
        if (FILL && *fmask_s) {
            // device fill: every CTA copies its share of each missing record from the fill source
            // into its slot; after a grid barrier the slots and the table point at them
            const uint32_t fm = *fmask_s;
            const size_t rb = 3 * matrix_bytes(a.I, H);
            const size_t S = align_up((rb + gridDim.x - 1) / gridDim.x, 16);
            const size_t lo = (size_t)blockIdx.x * S, hi = lo + S < rb ? lo + S : rb;
            for (int k = 0; k < a.K; ++k) {
                if (!((fm >> k) & 1u) || lo >= hi) continue;
                const size_t at = (size_t)l * E + fid_s[k];
                copy16_batched(reinterpret_cast<uint4 *>(a.fill_dst[at] + lo),
                               reinterpret_cast<const uint4 *>(a.fill_src[at] + lo), (uint32_t)((hi - lo) / 16));
            }
            if (!grid_sync(a.ctr, target, ok_s, a.ctrl, cap_grid)) { failed = true; break; }
            if (threadIdx.x < (unsigned)a.K && ((fm >> threadIdx.x) & 1u)) {
                const size_t at = (size_t)l * E + fid_s[threadIdx.x];
                const uint64_t d = a.fill_dst[at];
                slots_s[threadIdx.x] = d;
                if (blockIdx.x == 0) {
                    a.table_w[at] = d;
                    a.slots[(size_t)l * a.K + threadIdx.x] = d;
                    atomicAdd(a.filled, 1u);
                }
            }
            cta_sync();
        }
        // after a device fill the producer warp issues the gate/up copies from the new slots
        if (warp == kStProducer && !early) issue_gu(slots_s[C.ka], slots_s[C.kb]);
        // the computing warps start once every copy is issued: issued under their load the
        // copies take about three times longer
        cta_sync();
        ex_issued = true;

        // ---------------- C: gate/up + SwiGLU of this CTA's pairs ----------------
        if (C.p1 > C.p0) {
            const int p0 = C.p0, p1 = C.p1, n0 = C.n0, n1 = C.n1, rowb = C.rowb;
            const uint8_t *gtiles = smem + C.o_gu;
            float *part = reinterpret_cast<float *>(smem + C.o_part);
            const int half = warp % SPLIT, team = warp / SPLIT;
            constexpr int kTeams = kStWarps / SPLIT;
            const int c0 = half * (H / SPLIT) + lane * 8 * GPL;
            unsigned long long xv[4 * GPL];  // the lane's inputs as packed f32 pairs
            {
                const float r = *scale_s;
                const float4 *xt_s = reinterpret_cast<const float4 *>(smem + C.o_xt);
#pragma unroll
                for (int q = 0; q < 2 * GPL; ++q) {
                    const float4 v = xt_s[(half * 2 * GPL + q) * 32 + (lane ^ q)];
                    pack4(make_float4(v.x * r, v.y * r, v.z * r, v.w * r), &xv[2 * q]);
                }
            }
            const uint4 *tabc = tab + (lane & (kTabCopies - 1));
            const int gl = c0 / 8, boff = (gl >> 5) * kBlockBytes, g0 = gl & 31;
            unsigned ready = 0;
            bool to = false;
            auto locate = [&](int p, const uint8_t *&gb, const uint8_t *&ub) {
                const int seg = p - p0 < n0 ? 0 : 1;
                const int r = seg == 0 ? p - p0 : p - p0 - n0;
                const int n = seg == 0 ? n0 : n1;
                int ch = 0;
                while (ch + 1 < kStGuChunks && r >= ((n / U) * (ch + 1) / kStGuChunks) * U) ++ch;
                const int bi = seg * kStGuChunks + ch;
                if (!(ready & (1u << bi))) {
                    if (!mbar_wait_warp(&bar_gu[bi], ph, cap_wait)) to = true;
                    ready |= 1u << bi;
                }
                gb = gtiles + (seg == 0 ? 0 : 2 * (size_t)n0 * rowb) + (size_t)r * rowb + boff;
                ub = gb + (size_t)n * rowb;
            };
            for (int p = p0 + team; p < p1; p += 2 * kTeams) {
                const int q = p + kTeams;  // second row pair in flight
                const uint8_t *gb, *ub, *gb2 = nullptr, *ub2 = nullptr;
                locate(p, gb, ub);
                if (q < p1) locate(q, gb2, ub2);
                if (to) break;
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
            if (to) failed = true;
        }
        // The last warp (whose team has no more rows than any other) then issues the down rows
        // of the K experts, which D needs after the next grid barrier, the next layer's router
        // columns and an L2 prefetch of its residency row (read once per token, it would come
        // from HBM).
        if (warp == kStProducer && !failed) {
            fence_proxy_async_smem();
            if (FILL) asm volatile("fence.proxy.async.global;" ::: "memory");
            const int K = a.K, I = a.I, nq = C.nq;
            const size_t matb = matrix_bytes(I, H);
            if (nq > 0) {
                const uint32_t bytes = (uint32_t)matrix_bytes(nq, I);
                if (lane == 0) mbar_arrive_expect_tx(bar_dn, bytes * K);
                __syncwarp();
                if (lane < K)
                    bulk_g2s(smem + C.o_dn + (size_t)lane * C.dtileb,
                             reinterpret_cast<const uint8_t *>(slots_s[lane]) + 2 * matb + matrix_bytes(C.q0, I), bytes,
                             bar_dn);
            }
            if (threadIdx.x == kColThread) {
                if (!last && nq > 0) issue_cols(i + 1);
                if (!last && tab_smem) issue_tab(i + 1);  // the next layer's residency row
                *iss_s = (nq > 0 ? 1 : 0) | (!last && nq > 0 ? 2 : 0) | (!last && tab_smem ? 4 : 0);
            }
            __syncwarp();
        }
        failed = cta_sync_or(failed) != 0;
        if (*iss_s & 2) rc_pend = i + 1;
        if (*iss_s & 4) tab_pend = i + 1;
        if (failed) break;
        {
            const int p0 = C.p0, np = C.p1 - C.p0;
            const float *part = reinterpret_cast<const float *>(smem + C.o_part);
            for (int t = threadIdx.x; t < np; t += kStThreads) __stcg(a.h + p0 + t, swiglu_part<SPLIT>(part + 4 * t));
        }
        if (!grid_sync(a.ctr, target, ok_s, a.ctrl, cap_grid)) { failed = true; break; }

        // ---------------- D: down rows of every expert, ordered combine, residual ----------------
        // acc[i & 1] was read by every CTA in B; it takes the sums of layer index i + 2 next
        if (blockIdx.x == 0) {
            for (int j = threadIdx.x; j < E; j += kStThreads) __stcg(a.acc + (size_t)(i & 1) * E + j, 0ll);
            if (threadIdx.x == 0) __stcg(a.ss + (i & 1), 0ll);
        }
        // the renormalised weights, needed first by the combine (off the path from the
        // selection to the expert copies); by a warp with the smaller share of the h staging
        if (warp == kStProducer - 1) {
            const int K = a.K;
            const float w = topk_weight(lane < K ? sv_s[lane] : 0.f, K);
            if (lane < K) {
                w_s[lane] = w;
                if (blockIdx.x == 0) a.weights[(size_t)l * K + lane] = w;
            }
            __syncwarp();
        }
        // The producer warp (idle in D when K > 8) meanwhile selects the pre-gated prediction of
        // the next layer's experts and prefetches this CTA's slice of their records into L2
        // ("Red Lite dev23", "What changed": pre-gated expert prefetch).
        if (pregate && !last && warp == kStProducer) {
            const int P = a.pregate;
            const float rs = *scale_s;
            const long long *ap = a.acc_pg + (size_t)(i & 1) * E;
            const float *b1 = a.bias ? a.bias + (size_t)(l + 1) * E : nullptr;
            int pid;
            float pval;
            warp_topk_by<kStCand, kStPredMax>(
                [&](int e) { return e < E ? order_key(fmaf(fixed_value(__ldcg(ap + e)), rs, b1 ? b1[e] : 0.f)) : 0u; },
                P, pid, pval);
            uint64_t pslot = 0;
            if (lane < P) {
                pred_s[lane] = pid;
                pslot = __ldcg(a.table + (size_t)(l + 1) * E + pid);
            }
            const size_t rec = 3 * matrix_bytes(a.I, H);
            const size_t total = (size_t)P * rec;
            const size_t S = align_up((total + gridDim.x - 1) / gridDim.x, 16);
            const size_t lo = (size_t)blockIdx.x * S, hi = lo + S < total ? lo + S : total;
            if (lane < P && pslot != 0 && (pslot & 15) == 0) {
                const size_t r0 = (size_t)lane * rec, r1 = r0 + rec;
                const size_t b0 = lo > r0 ? lo : r0, b1 = hi < r1 ? hi : r1;
                if (b1 > b0) prefetch_l2_bulk(reinterpret_cast<const uint8_t *>(pslot) + (b0 - r0), (uint32_t)(b1 - b0));
            }
            __syncwarp();
        }
        {
            // every group of LPR lanes owns one expert (group g: expert g % K) and every
            // (K)-th of its rows; a warp runs as many passes as its busier half needs, so the
            // shuffles of a row's reduction always see the whole warp
            const int nq = C.nq, K = a.K;
            // h of all K experts into shared memory, once per CTA, lane-transposed: float4 q of
            // lane sl of a row group (h_k[8 DGPL sl + 4 q ...]) sits at [k][q][sl ^ q], so that a
            // group's reads (fixed q, 16 or 32 consecutive sl) and the staging writes (8
            // consecutive q of one sl per quarter warp) both spread over all banks.  The global
            // reads are coalesced.
            if (nq > 0) {
                const int I = a.I, f4 = I / 4;
                float4 *h_s = reinterpret_cast<float4 *>(smem + C.o_h);
                const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
                for (int d = threadIdx.x; d < K * f4; d += kStThreads) {
                    const int k = d / f4, r = d % f4, sl = r / (2 * DGPL), q = r % (2 * DGPL);
                    h_s[k * f4 + q * LPR + (sl ^ q)] = __ldcg(h4 + d);
                }
                cta_sync();
            }
            if (nq > 0) {
                constexpr int kNG = kStThreads / LPR;  // lane groups in the CTA
                const int g = threadIdx.x / LPR, sl = lane % LPR;
                const int k = g % K, jg = g / K, ngk = (kNG - k + K - 1) / K;
                const int mine = jg < nq ? (nq - jg + ngk - 1) / ngk : 0;
                const int trips = (int)__reduce_max_sync(kFull, (unsigned)mine);
                const int I = a.I, dmax = C.dmax;
                unsigned long long hv[4 * DGPL];  // h of the lane's expert as packed f32 pairs
                const float4 *h_s = reinterpret_cast<const float4 *>(smem + C.o_h) + (size_t)k * (I / 4);
#pragma unroll
                for (int q = 0; q < 2 * DGPL; ++q) pack4(h_s[q * LPR + (sl ^ q)], &hv[2 * q]);
                if (trips > 0 && !mbar_wait_warp(bar_dn, ph, cap_wait)) {
                    failed = true;
                } else {
                    const uint4 *tabc = tab + (lane & (kTabCopies - 1));
                    const uint8_t *tile = smem + C.o_dn + (size_t)k * C.dtileb;
                    float *o_s = reinterpret_cast<float *>(smem + C.o_o);
                    for (int t = 0; t < trips; ++t) {
                        const int rr = jg + t * ngk;
                        const bool real = rr < nq;
                        const float o = down_row<DGPL, LPR>(tile, real ? rr : 0, I, sl, hv, tabc);
                        if (real && sl == 0) o_s[k * dmax + rr] = o;
                        __syncwarp();
                    }
                }
            }
        }
        failed = cta_sync_or(failed) != 0;
        if (failed) break;
        ex_issued = false;
        if (threadIdx.x == 0) *iss_s = 0;  // the down rows have landed (waited above)
        if ((int)threadIdx.x < C.nq) {
            const int r = C.q0 + threadIdx.x;
            const float *o_s = reinterpret_cast<const float *>(smem + C.o_o);
            float *xq = reinterpret_cast<float *>(smem + C.o_xq);  // this CTA's slice of x_l
            const float acc = ordered_combine(w_s, o_s + threadIdx.x, C.dmax, a.K);
            if (a.y) {
                a.y[r] = acc;  // a single layer (nl = 1): the loop ends below
            } else {
                const float xv = xq[threadIdx.x] + acc;
                __stcg(a.x + r, xv);
                xq[threadIdx.x] = xv;
            }
        }
        if (last) break;
        // the next layer's router dots on this CTA's slice of x_{l+1}
        if (warp == 0 && C.nq > 0 && !mbar_spin_warp(bar_rc, (uint32_t)((i + 1) & 1), cap_spin)) failed = true;
        failed = cta_sync_or(failed) != 0;
        if (failed) break;
        rc_pend = -1;
        add_partials(i + 1);
        if (!grid_sync(a.ctr, target, ok_s, a.ctrl, cap_grid)) { failed = true; break; }
    }
    // ---- exit: no copy into this CTA's shared memory may still be in flight ----
    if (threadIdx.x == 0) {
        bool drained = true;
        if (rc_pend >= 0) drained &= mbar_wait(bar_rc, (uint32_t)(rc_pend & 1), cap_wait);
        if (tab_pend >= 0) drained &= mbar_wait(bar_tab, (uint32_t)(tab_pend & 1), cap_wait);
        if (*iss_s & 1) drained &= mbar_wait(bar_dn, ph, cap_wait);
        if (ex_issued) {
            for (int bi = 0; bi < 2 * kStGuChunks; ++bi) {
                const int seg = bi / kStGuChunks, ch = bi % kStGuChunks;
                if (C.p1 > C.p0 && gu_cut(C, U, seg, ch + 1) > gu_cut(C, U, seg, ch))
                    drained &= mbar_wait(&bar_gu[bi], ph, cap_wait);
            }
        }
        if (!drained) dev_error(a.ctrl, RL_DEVERR_WAIT_TIMEOUT);
    }
    cta_sync();
}


template <int NV, int GPL, int SPLIT, int DGPL, int LPR, bool FILL>
static rl_status launch_stack(StackArgs a, cudaStream_t s) {
    auto kern = stack_kernel<NV, GPL, SPLIT, DGPL, LPR, FILL>;
    const int G = sm_count();
    const StLayout lay(a.H, a.E, a.K, a.I, G, a.pregate > 0);
    if (lay.total > 227 * 1024 || a.E > kStThreads || G > kStMaxGrid || lay.rmax > a.I || lay.dmax > 256 ||
        kStWarps / a.K < 1)
        return fail(RL_ERR_UNSUPPORTED, "moe_decode_stack: shape does not fit one CTA per SM (H=%d E=%d K=%d I=%d)",
                    a.H, a.E, a.K, a.I);
    // The router as a [n_layers * E][H] f32 matrix; a box is rc_rows(E) rows x dmax columns.
    // The encoded map and the occupancy check are kept per device and router (a single-layer
    // launch is short enough that recomputing them on the host every time shows in the rate).
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int, int, int, int>, CUtensorMap> maps;  // every input of the map
    static std::map<std::tuple<int, const void *, size_t>, int> occs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "moe_decode_stack: cudaGetDevice: %s", cudaGetErrorString(e));
    {
        std::lock_guard<std::mutex> lk(mu);
        const auto mk = std::make_tuple(dev, (const void *)a.W, a.H, a.E, a.n_layers, lay.dmax);
        auto it = maps.find(mk);
        if (it != maps.end()) {
            a.wmap = it->second;
        } else {
            PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
            if (!enc) return fail(RL_ERR_CUDA, "moe_decode_stack: cuTensorMapEncodeTiled unavailable");
            const cuuint64_t gdim[2] = {(cuuint64_t)a.H, (cuuint64_t)a.n_layers * a.E};
            const cuuint64_t gstride[1] = {(cuuint64_t)a.H * sizeof(float)};
            const cuuint32_t box[2] = {(cuuint32_t)lay.dmax, (cuuint32_t)rc_rows(a.E)};
            const cuuint32_t estride[2] = {1, 1};
            CUresult cr = enc(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.W), gdim, gstride, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (cr != CUDA_SUCCESS)
                return fail(RL_ERR_UNSUPPORTED, "moe_decode_stack: router tensor map rejected (error %d, box %d x %d)",
                            (int)cr, lay.dmax, rc_rows(a.E));
            if (maps.size() >= 64) maps.clear();  // routers of models since freed
            maps[mk] = a.wmap;
        }
    }
    rl_status st = allow_smem((const void *)kern, lay.total);
    if (st != RL_OK) return st;
    int occ = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        const auto ok = std::make_tuple(dev, (const void *)kern, lay.total);
        auto it = occs.find(ok);
        if (it != occs.end()) {
            occ = it->second;
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kStThreads, lay.total);
            if (e != cudaSuccess) occ = 0;
            else occs[ok] = occ;
        }
    }
    if (occ < 1) return fail(RL_ERR_UNSUPPORTED, "moe_decode_stack: no SM can hold the %zu B CTA", lay.total);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kStThreads);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "moe_decode_stack: launch failed: %s", cudaGetErrorString(e));
    return RL_OK;
}

template <int NV, int GPL, int SPLIT, bool FILL>
static rl_status launch_stack_i(const StackArgs &a, cudaStream_t s) {
    switch (a.I) {
        case 128: return launch_stack<NV, GPL, SPLIT, 1, 16, FILL>(a, s);
        case 256: return launch_stack<NV, GPL, SPLIT, 1, 32, FILL>(a, s);
        case 512: return launch_stack<NV, GPL, SPLIT, 4, 16, FILL>(a, s);
        case 1024: return launch_stack<NV, GPL, SPLIT, 4, 32, FILL>(a, s);
        default: return launch_stack<NV, GPL, SPLIT, 8, 32, FILL>(a, s);
    }
}

// every shape, one variant
template <bool FILL>
static rl_status launch_stack_any(const StackArgs &a, cudaStream_t s) {
    switch (a.H) {
        case 256: return launch_stack_i<2, 1, 1, FILL>(a, s);
        case 512: return launch_stack_i<4, 2, 1, FILL>(a, s);
        case 1024: return launch_stack_i<8, 2, 2, FILL>(a, s);
        default: return launch_stack_i<16, 4, 2, FILL>(a, s);
    }
}

// the device-fill variants, compiled in their own translation unit (stack_fill.cu)
rl_status launch_stack_fill(const StackArgs &a, cudaStream_t s);

}  // namespace rl
