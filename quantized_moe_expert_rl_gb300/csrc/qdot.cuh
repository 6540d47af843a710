// qdot.cuh - in-register decode of the 66-byte codebook blocks for the CUDA-core GEMVs.
//
// The 256 x 8 int8 codebook is converted once per CTA into a table of bf16 pairs (every
// int8 value is exact in bf16): entry idx = 4 words, word i = bf16(g[2i]) | bf16(g[2i+1]) << 16.
// The table is stored 8 times, interleaved so that entry e of copy c sits at 16-byte slot
// e*8 + c; lane L reads copy L & 7, so the 8 lanes of each quarter-warp phase of a 128-bit
// shared load always hit 8 different bank quads, whatever indices they look up.
//
// Signs: one multiply and one LOP3 sign a pair word (group_fma2).  The two bf16 halves become
// f32 by a shift (low) and a mask (high), and a packed f32x2 FMA accumulates both.
#pragma once
#include "rl_common.cuh"

namespace rl {

constexpr int kTabCopies = 8;
constexpr int kTabBytes = 256 * 16 * kTabCopies;  // 32 KB

__device__ __forceinline__ uint32_t bf16_bits(int v) {
    // exact for |v| <= 256: bf16 has an 8-bit significand
    return __float_as_uint((float)v) >> 16;
}

// Build the replicated pair table from the int8 codebook with the whole CTA.  The 2 KB
// codebook is first staged through `stage` (>= 2 KB of shared memory, reused afterwards) with
// one coalesced load per thread, then expanded; ends with __syncthreads().
__device__ __forceinline__ void build_pair_table(uint4 *tab, const int8_t *__restrict__ codebook, uint2 *stage) {
    (void)stage;
    // each entry is converted once (256 threads) and written to its 8 copies
    for (int e = threadIdx.x; e < 256; e += blockDim.x) {
        const uint2 raw = reinterpret_cast<const uint2 *>(codebook)[e];
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t word = p < 2 ? raw.x : raw.y;
            const int g0 = (int8_t)((word >> (16 * (p & 1))) & 0xffu);
            const int g1 = (int8_t)((word >> (16 * (p & 1) + 8)) & 0xffu);
            w[p] = bf16_bits(g0) | (bf16_bits(g1) << 16);
        }
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int c = 0; c < kTabCopies; ++c)  // rotated so one store instruction hits 8 bank quads
            tab[e * kTabCopies + ((c + threadIdx.x) & (kTabCopies - 1))] = v;
    }
    __syncthreads();
}

__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
    return (unsigned long long)lo | ((unsigned long long)hi << 32);
}
__device__ __forceinline__ float hsum2(unsigned long long a) {
    return __uint_as_float((uint32_t)a) + __uint_as_float((uint32_t)(a >> 32));
}

// acc += sum_{j<8} grid[idx][j] * (+-1)_j * x[j] for one group; `gs` = (idx | sign << 8),
// `x` = 4 packed f32 pairs (x0,x1) (x2,x3) (x4,x5) (x6,x7), `tabc` = this lane's table copy,
// `acc` = packed (even, odd) accumulators.  The signs of pair word i come from one multiply:
// s * (2^(15-2i) + 2^(30-2i)) puts bit 2i of s at bit 15 and bit 2i+1 at bit 31 (the two
// shifted copies of the 8-bit s do not overlap, so nothing carries).  About 25 instructions per
// 8 weights; measured 8% faster than shifts for the signs and scalar FMAs.
__device__ __forceinline__ unsigned long long group_fma2(uint32_t gs, const unsigned long long *x, const uint4 *tabc,
                                                         unsigned long long acc) {
    const uint4 q = tabc[(gs & 0xffu) * kTabCopies];
    const uint32_t s = gs >> 8;
    const uint32_t w0 = q.x ^ ((s * 0x40008000u) & 0x80008000u), w1 = q.y ^ ((s * 0x10002000u) & 0x80008000u);
    const uint32_t w2 = q.z ^ ((s * 0x04000800u) & 0x80008000u), w3 = q.w ^ ((s * 0x01000200u) & 0x80008000u);
    acc = ffma2(pack2(w0 << 16, w0 & 0xffff0000u), x[0], acc);
    acc = ffma2(pack2(w1 << 16, w1 & 0xffff0000u), x[1], acc);
    acc = ffma2(pack2(w2 << 16, w2 & 0xffff0000u), x[2], acc);
    acc = ffma2(pack2(w3 << 16, w3 & 0xffff0000u), x[3], acc);
    return acc;
}
// 4 f32 values -> 2 packed pairs
__device__ __forceinline__ void pack4(float4 v, unsigned long long *p) {
    p[0] = pack2(__float_as_uint(v.x), __float_as_uint(v.y));
    p[1] = pack2(__float_as_uint(v.z), __float_as_uint(v.w));
}

// RMSNorm scale 1/sqrt(mean(x^2) + eps) with an exact, order-free sum of squares, so that
// every kernel that normalises a row (whole or split between CTAs) gets the same bits.  The
// squares of each group of 8 consecutive values are added in the fixed tree
// ((x0^2 + x1^2) + (x2^2 + x3^2)) + ((x4^2 + x5^2) + (x6^2 + x7^2)) in f32 without
// contraction; each group sum is rounded to a multiple of 2^-30 and the groups are added as
// 64-bit integers (exact, so any split of the groups gives the same total).  A group sum at or
// above 2^25 (|x| beyond about 1400) or NaN is outside the range: it counts as 2^25 and the
// caller is told (RL_DEVERR_RANGE where it has a control block).
constexpr float kSqScale = 1073741824.0f;          // 2^30
constexpr float kSqInv = 9.313225746154785e-10f;   // 2^-30
constexpr float kSqMax = 33554432.0f;              // 2^25

__device__ __forceinline__ float sq8(float4 a, float4 b) {
    const float p = __fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)),
                              __fadd_rn(__fmul_rn(a.z, a.z), __fmul_rn(a.w, a.w)));
    const float q = __fadd_rn(__fadd_rn(__fmul_rn(b.x, b.x), __fmul_rn(b.y, b.y)),
                              __fadd_rn(__fmul_rn(b.z, b.z), __fmul_rn(b.w, b.w)));
    return __fadd_rn(p, q);
}
// The same group sum when lane t of an aligned group of 8 lanes holds value t: the shuffle
// tree pairs the same terms (and f32 addition is commutative), so every lane of the group
// returns sq8's bits.  Call with the whole warp.
__device__ __forceinline__ float sq8_lanes(float v) {
    float s = __fmul_rn(v, v);
    s = __fadd_rn(s, __shfl_xor_sync(kFull, s, 1));
    s = __fadd_rn(s, __shfl_xor_sync(kFull, s, 2));
    s = __fadd_rn(s, __shfl_xor_sync(kFull, s, 4));
    return s;
}
__device__ __forceinline__ long long sq_fixed(float s, bool &range) {
    if (!(s < kSqMax)) {
        range = true;
        s = kSqMax;
    }
    return float_to_ll(s * kSqScale);
}
__device__ __forceinline__ float rms_scale_from(long long ss, int H, float eps) {
    return 1.0f / sqrtf(ll_to_float(ss) * kSqInv / (float)H + eps);
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// The scale of H values (H a multiple of 256) by ONE warp: lane L takes the groups L, L + 32,
// ...  Returns the scale in every lane; *range (optional) is set in every lane when a group
// was out of range.
__device__ __forceinline__ float rms_scale_warp(const float *__restrict__ x, int H, float eps, bool *range = nullptr) {
    const int lane = threadIdx.x & 31;
    long long acc = 0;
    bool rg = false;
    for (int g = lane; g < H / 8; g += 32) {
        const float4 a = *reinterpret_cast<const float4 *>(x + 8 * g);
        const float4 b = *reinterpret_cast<const float4 *>(x + 8 * g + 4);
        acc += sq_fixed(sq8(a, b), rg);
    }
    acc = warp_sum_ll(acc);
    const bool any = __any_sync(kFull, rg);
    if (range) *range = any;
    return rms_scale_from(acc, H, eps);
}

// ---- programmatic dependent launch ---------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace rl
