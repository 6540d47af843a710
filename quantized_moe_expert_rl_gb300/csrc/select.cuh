// select.cuh - top-k selection of one token's router logits by one warp, with the
// renormalised weights ("Red Lite dev21 - GPU-routed decode", "What changed": rl_route picks
// the top-k by logit, ties to the lower index, and renormalises the weights over the
// selection).  Shared by rl_route and the fused decode stack so both select identically.
//
// Lane l holds experts l*C .. l*C+C-1 (C = candidates per lane), so a lower lane always holds
// lower expert indices.  Keys are the f32 logits mapped to order-preserving uint32 after
// folding -0.0 into +0.0 (so the two compare equal); key 0 is below every finite value and
// marks a taken or absent candidate.  Each round takes the warp maximum with redux.sync; among
// equal keys the lowest lane wins, and inside a lane the first (lowest) index wins, so ties go
// to the lower expert index.
#pragma once
#include "rl_common.cuh"

namespace rl {

constexpr int kMaxK = 16;  // largest top-k the library accepts

// A NaN logit gets key 0: it ranks below every number, like an absent candidate (the callers
// raise RL_DEVERR_NAN for it).
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v + 0.0f);  // -0.0 + 0.0 = +0.0
    if (v != v) return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// After the call lane r < K holds the r-th selected expert (my_id) and its logit (my_val).
// key_of(e) gives the key of expert e (0 for an absent one), for e < 32 * C.  K <= MAXK <= 32.
template <int C, int MAXK = kMaxK, class KeyOf>
__device__ __forceinline__ void warp_topk_by(KeyOf key_of, int K, int &my_id, float &my_val) {
    const int lane = threadIdx.x & 31;
    uint32_t key[C];
    uint32_t best = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        key[i] = key_of(lane * C + i);
        if (key[i] > best) { best = key[i]; bi = i; }
    }
    my_id = 0;
    my_val = 0.f;
#pragma unroll
    for (int r = 0; r < MAXK; ++r) {
        if (r >= K) break;
        const uint32_t m = __reduce_max_sync(kFull, best);
        const int wl = __ffs(__ballot_sync(kFull, best == m)) - 1;
        const int wi = __shfl_sync(kFull, bi, wl);
        if (lane == r) { my_id = wl * C + wi; my_val = key_value(m); }
        if (lane == wl) {  // the winner drops its candidate and finds its next best
            best = 0u;
            bi = 0;
#pragma unroll
            for (int i = 0; i < C; ++i) {
                if (i == wi) key[i] = 0u;
                if (key[i] > best) { best = key[i]; bi = i; }
            }
        }
        __syncwarp();  // rejoin before the next round's votes (see cta_sync)
    }
}

// warp_topk_by on E logits read through L2 (they may come from other CTAs); true in every lane
// when one of the logits was NaN
template <int C>
__device__ __forceinline__ bool warp_topk(const float *lg, int E, int K, int &my_id, float &my_val) {
    bool nan = false;
    warp_topk_by<C>(
        [&](int e) {
            if (e >= E) return 0u;
            const float v = __ldcg(lg + e);
            nan |= v != v;
            return order_key(v);
        },
        K, my_id, my_val);
    return __any_sync(kFull, nan);
}

// w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), the sum taken in selection order; lane k < K
// gets w_k (other lanes 0).
__device__ __forceinline__ float topk_weight(float my_val, int K) {
    const int lane = threadIdx.x & 31;
    const float l0 = __shfl_sync(kFull, my_val, 0);
    const float ex = lane < K ? expf(my_val - l0) : 0.f;
    float tot = 0.f;
    // unrolled to the largest K (16) with the adds predicated: a loop over a run-time K with a
    // shuffle in its body ran about ten times slower
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        const float v = __shfl_sync(kFull, ex, k);
        if (k < K) tot += v;
    }
    return lane < K ? ex / tot : 0.f;
}

// Full rl_route selection for one token: ids, weights, slots, miss count and flag.
template <int C>
__device__ __forceinline__ void warp_select(const float *lg, const uint64_t *__restrict__ table_row,
                                            int32_t *ids, float *weights, uint64_t *slots, uint32_t *miss_l,
                                            int32_t *ctrl, int layer, int E, int K) {
    const int lane = threadIdx.x & 31;
    int my_id;
    float my_val;
    if (warp_topk<C>(lg, E, K, my_id, my_val) && lane == 0) dev_error(ctrl, RL_DEVERR_NAN);
    const float w = topk_weight(my_val, K);
    uint64_t slot = 1;
    if (lane < K) {
        ids[lane] = my_id;
        weights[lane] = w;
        slot = table_row[my_id];
        slots[lane] = slot;
    }
    __syncwarp();
    const int nmiss = __popc(__ballot_sync(kFull, lane < K && slot == 0));
    if (lane == 0 && nmiss > 0) {
        atomicAdd(miss_l, (uint32_t)nmiss);
        atomicMin(ctrl, layer);
    }
}

}  // namespace rl

namespace rl {

// (ka, ia) comes before (kb, ib) in the selection order: larger key, then lower index
__device__ __forceinline__ bool precedes(uint32_t ka, int ia, uint32_t kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Top-k of up to 32 * NW logits with NW warps of one CTA (the fused decode stack runs it in
// every CTA), in few dependent steps.  Thread 32w + lane passes `key`, the key of expert
// 32w + lane (0 when absent; the threads of warps >= NW pass 0).  Let m_w be
// the largest key of warp w and T the K-th largest of the m_w: the
// K warps holding the K largest maxima give K keys >= T, so the K-th largest key overall is
// >= T and every key of the top-K is >= T.  The keys >= T (usually a few tens) are gathered and
// each is ranked exactly against the others in the order (logit descending, index ascending);
// the K first are the selection, the same as warp_topk's.  cand_*: shared scratch of 32 * NW
// entries; wm_s: NW words; sel: K entries; cnt_s: one word.  Lane r < K of every warp ends
// with the r-th selection; the CTA is converged on return.  K <= NW.
template <int NW>
__device__ __forceinline__ void cta_topk_thr(uint32_t key, const uint64_t *__restrict__ table_row, int E, int K,
                                             uint32_t *cand_key, int *cand_id, uint64_t *cand_slot,
                                             uint32_t *wm_s, int *sel, int *cnt_s, int &my_id, float &my_val,
                                             uint64_t &my_slot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = warp * 32 + lane;
    if (warp >= NW || e >= E) key = 0u;
    if (threadIdx.x == 0) *cnt_s = 0;
    if (warp < NW) {
        const uint32_t m = __reduce_max_sync(kFull, key);
        if (lane == 0) wm_s[warp] = m;
    }
    cta_sync();
    if (warp < NW) {
        // T = the K-th largest warp maximum (ties by warp index, which only fixes who holds it)
        const uint32_t mj = lane < NW ? wm_s[lane] : 0u;
        int rank = 0;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t mi = wm_s[i];
            rank += (mi > mj || (mi == mj && i < lane)) ? 1 : 0;
        }
        const int who = __ffs(__ballot_sync(kFull, lane < NW && rank == K - 1)) - 1;
        const uint32_t T = __shfl_sync(kFull, mj, who);
        const bool cand = e < E && key >= T;
        const unsigned mask = __ballot_sync(kFull, cand);
        int base = 0;
        if (lane == 0 && mask) base = atomicAdd(cnt_s, __popc(mask));
        __syncwarp();
        base = __shfl_sync(kFull, base, 0);
        if (cand) {
            const int at = base + __popc(mask & ((1u << lane) - 1u));
            cand_key[at] = key;
            cand_id[at] = e;
            cand_slot[at] = __ldcg(table_row + e);
        }
    }
    cta_sync();
    const int n = *cnt_s;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
        const uint32_t kc = cand_key[c];
        const int ic = cand_id[c];
        int r = 0;
#pragma unroll 4
        for (int j = 0; j < n; ++j) r += precedes(cand_key[j], cand_id[j], kc, ic) ? 1 : 0;
        if (r < K) sel[r] = c;
    }
    cta_sync();
    my_id = 0;
    my_val = 0.f;
    my_slot = 0;
    if (lane < K) {
        const int c = sel[lane];
        my_id = cand_id[c];
        my_val = key_value(cand_key[c]);
        my_slot = cand_slot[c];
    }
    __syncwarp();
}

}  // namespace rl

namespace rl {

// Top-k of up to 512 keys by ONE warp, in a few dependent steps, so that every warp of a CTA
// can select on its own with no CTA barrier after the keys are written.  keys_t holds the key
// of expert e at [(e % 16) * 32 + e / 16] (0 for absent experts and for e >= E), so lane L
// reads the keys of experts 16 L .. 16 L + 15 with conflict-free loads and lower lanes hold
// lower indices.  Let m_L be lane L's largest key and T the K-th largest of the 32 m_L: the K
// lanes holding the K largest give K keys >= T, so every key of the top-K is >= T.  The keys
// >= T (a few tens at most, usually) are gathered into the warp's scratch and each is ranked
// exactly against the others in the order (logit descending, index ascending); with more than
// 32 candidates (heavy ties) K rounds of warp arg-max take over.  The selection equals
// warp_topk's.  Scratch: ck[32], ci[32], sel[kMaxK] of this warp.  Lane r < K ends with the
// r-th selection; the warp is converged on return.
__device__ __forceinline__ void warp_topk_thr(const uint32_t *keys_t, int E, int K, uint32_t *ck, int *ci, int *sel,
                                              int &my_id, float &my_val) {
    const int lane = threadIdx.x & 31;
    uint32_t k[16];
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        k[j] = keys_t[j * 32 + lane];
        m = k[j] > m ? k[j] : m;
    }
    int rank = 0;  // rank of m among the lane maxima (ties by lane)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t mj = __shfl_sync(kFull, m, j);
        rank += (mj > m || (mj == m && j < lane)) ? 1 : 0;
    }
    const uint32_t T = __shfl_sync(kFull, m, __ffs(__ballot_sync(kFull, rank == K - 1)) - 1);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) cnt += (16 * lane + j < E && k[j] >= T) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += u;
    }
    const int n = __shfl_sync(kFull, incl, 31);
    my_id = 0;
    my_val = 0.f;
    if (n <= 32) {
        int at = incl - cnt;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (16 * lane + j < E && k[j] >= T) {
                ck[at] = k[j];
                ci[at] = 16 * lane + j;
                ++at;
            }
        __syncwarp();
        // lane c holds candidate c and ranks it against the others through shuffles
        const uint32_t kc = lane < n ? ck[lane] : 0u;
        const int ic = lane < n ? ci[lane] : 0x7fffffff;
        int r = 0;
#pragma unroll
        for (int d = 0; d < 32; ++d) {
            const uint32_t kd = __shfl_sync(kFull, kc, d);
            const int id = __shfl_sync(kFull, ic, d);
            r += (d < n && precedes(kd, id, kc, ic)) ? 1 : 0;
        }
        if (lane < n && r < K) sel[r] = lane;
        __syncwarp();
        if (lane < K) {
            const int c = sel[lane];
            my_id = ci[c];
            my_val = key_value(ck[c]);
        }
        __syncwarp();
    } else {
        warp_topk_by<16>([&](int e) { return e < E ? keys_t[(e & 15) * 32 + (e >> 4)] : 0u; }, K, my_id, my_val);
    }
}

// RMSNorm scale of x (H = NV * 128 values) read through L2 (x written by other CTAs of the
// same launch), every load issued before the arithmetic: the arithmetic and order of
// rms_scale_warp exactly, so every path normalises identically.
template <int NV>
__device__ __forceinline__ float rms_scale_warp_cg(const float *x, float eps) {
    const int lane = threadIdx.x & 31;
    float4 v[NV];
#pragma unroll
    for (int m = 0; m < NV; ++m) v[m] = __ldcg(reinterpret_cast<const float4 *>(x + lane * 4 + 128 * m));
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int m = 0; m < NV; ++m) {
        a0 = fmaf(v[m].x, v[m].x, a0); a1 = fmaf(v[m].y, v[m].y, a1); a2 = fmaf(v[m].z, v[m].z, a2); a3 = fmaf(v[m].w, v[m].w, a3);
    }
    float ss = warp_sum((a0 + a1) + (a2 + a3));
    return 1.0f / sqrtf(ss / (float)(NV * 128) + eps);
}

}  // namespace rl
