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

// The rounds of the selection on keys already in registers: key[i] is the key of expert
// lane * C + i (0 for an absent one).  After the call lane r < K holds the r-th selected expert
// (my_id) and its logit (my_val).  K <= MAXK <= 32.  Consumes `key`.
template <int C, int MAXK = kMaxK>
__device__ __forceinline__ void warp_topk_keys(uint32_t (&key)[C], int K, int &my_id, float &my_val) {
    const int lane = threadIdx.x & 31;
    uint32_t best = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < C; ++i)
        if (key[i] > best) { best = key[i]; bi = i; }
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

// The same with the keys given by key_of(e) for e < 32 * C.
template <int C, int MAXK = kMaxK, class KeyOf>
__device__ __forceinline__ void warp_topk_by(KeyOf key_of, int K, int &my_id, float &my_val) {
    const int lane = threadIdx.x & 31;
    uint32_t key[C];
#pragma unroll
    for (int i = 0; i < C; ++i) key[i] = key_of(lane * C + i);
    warp_topk_keys<C, MAXK>(key, K, my_id, my_val);
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

}  // namespace rl

namespace rl {

// Expert of key j of a lane in the layout the fused decode loads its logit accumulators in:
// chunk c = j / 2 covers experts [64 c, 64 c + 64), lane L holds experts 64 c + 2 L and
// 64 c + 2 L + 1 (one 16-byte load per lane and chunk, the warp's load contiguous), so that
// every CTA reads each 32-byte sector of the accumulators once.
__device__ __forceinline__ int sel_id(int lane, int j) { return 64 * (j >> 1) + 2 * lane + (j & 1); }

// Top-k of up to 512 keys by ONE warp from registers, in a few dependent steps: k[j] is the
// key of expert sel_id(lane, j) (0 for an absent expert and for ids >= E).  Let m_L be lane L's
// largest key and T the K-th largest of the 32 m_L: the K lanes holding the K largest give K
// keys >= T, so every key of the top-K is >= T.  The keys >= T (a few tens at most, usually)
// are gathered into the warp's scratch and each is ranked exactly against the others in the
// order (logit descending, index ascending); with more than 32 candidates (heavy ties) K
// rounds of exact warp arg-max over (key, index) take over.  The selection equals warp_topk's.
// The all-to-all comparisons read shared memory by broadcast (every lane the same word), not
// shuffles.  Scratch (this warp's, 8-byte aligned): wm[32] lane maxima, cand[32] (key, id)
// pairs, sel[kMaxK].  Lane r < K ends with the r-th selection; the warp is converged on return.
__device__ __forceinline__ void warp_topk_thr(const uint32_t (&k)[16], int E, int K, uint32_t *wm, uint2 *cand,
                                              int *sel, int &my_id, float &my_val) {
    const int lane = threadIdx.x & 31;
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = k[j] > m ? k[j] : m;
    wm[lane] = m;
    __syncwarp();
    int rank = 0;  // rank of m among the lane maxima (ties by lane)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4 v = reinterpret_cast<const uint4 *>(wm)[q];
        rank += (v.x > m || (v.x == m && 4 * q + 0 < lane)) ? 1 : 0;
        rank += (v.y > m || (v.y == m && 4 * q + 1 < lane)) ? 1 : 0;
        rank += (v.z > m || (v.z == m && 4 * q + 2 < lane)) ? 1 : 0;
        rank += (v.w > m || (v.w == m && 4 * q + 3 < lane)) ? 1 : 0;
    }
    const uint32_t T = wm[__ffs(__ballot_sync(kFull, rank == K - 1)) - 1];
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) cnt += (sel_id(lane, j) < E && k[j] >= T) ? 1 : 0;
    // exclusive prefix and total of cnt (<= 16: five bits) from one ballot per bit
    const unsigned lt = (1u << lane) - 1u;
    int pre = 0, n = 0;
#pragma unroll
    for (int bit = 0; bit < 5; ++bit) {
        const unsigned bb = __ballot_sync(kFull, (cnt >> bit) & 1);
        pre += __popc(bb & lt) << bit;
        n += __popc(bb) << bit;
    }
    my_id = 0;
    my_val = 0.f;
    if (n <= 32) {
        int at = pre;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (sel_id(lane, j) < E && k[j] >= T) cand[at++] = make_uint2(k[j], (uint32_t)sel_id(lane, j));
        __syncwarp();
        // lane c ranks candidate c against all n (broadcast reads)
        const uint2 me = lane < n ? cand[lane] : make_uint2(0u, 0x7fffffffu);
        int r = 0;
        for (int d = 0; d < n; ++d) {
            const uint2 o = cand[d];
            r += precedes(o.x, (int)o.y, me.x, (int)me.y) ? 1 : 0;
        }
        if (lane < n && r < K) sel[r] = lane;
        __syncwarp();
        if (lane < K) {
            const uint2 c = cand[sel[lane]];
            my_id = (int)c.y;
            my_val = key_value(c.x);
        }
        __syncwarp();
    } else {
        unsigned left = 0u;  // bit j: candidate j of this lane is an expert not yet taken
#pragma unroll
        for (int j = 0; j < 16; ++j) left |= (sel_id(lane, j) < E ? 1u : 0u) << j;
        for (int r = 0; r < K; ++r) {
            // this lane's first candidate in (key descending, index ascending) order
            uint32_t bk = 0u;
            int bi = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (((left >> j) & 1u) && precedes(k[j], sel_id(lane, j), bk, bi)) { bk = k[j]; bi = sel_id(lane, j); }
            // the warp's first: a strict total order, so every lane ends with the same winner
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint32_t ok = __shfl_xor_sync(kFull, bk, o);
                const int oi = __shfl_xor_sync(kFull, bi, o);
                if (precedes(ok, oi, bk, bi)) { bk = ok; bi = oi; }
            }
            if (lane == r) { my_id = bi; my_val = key_value(bk); }
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (sel_id(lane, j) == bi) left &= ~(1u << j);
        }
        __syncwarp();
    }
}

}  // namespace rl
