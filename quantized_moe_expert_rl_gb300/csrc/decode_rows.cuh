// decode_rows.cuh - the per-row arithmetic of the single-token expert GEMVs, shared by
// moe_decode's kernels and the fused decode stack so that both produce the same bits.
//
// The synthetic codebook format: a row is a run of 66-byte blocks of 256 values (fp16 scale d,
// then 32 groups of 8 values, each an index into the 256 x 8 grid plus a sign byte).  A lane
// decodes whole groups in registers (qdot.cuh) and the block scale multiplies the lane's
// partial sum once.
#pragma once
#include "qdot.cuh"

namespace rl {

// rows of the flat (expert, row) space handled together so that copies stay 16-byte multiples
__host__ __device__ inline int gu_unit(int H) { return H >= 2048 ? 1 : 2048 / H; }
// warps per row: wide rows are split in two halves so that a lane holds only 32 inputs
__host__ __device__ inline int gu_split(int H) { return H >= 1024 ? 2 : 1; }

// Partial (gate, up) dots of one lane for one row pair; xp = the lane's 8 GPL inputs as packed
// f32 pairs.
template <int GPL>
__device__ __forceinline__ void gu_row(const uint8_t *gb, const uint8_t *ub, int g0, const unsigned long long *xp,
                                       const uint4 *tabc, float &gv, float &uv) {
    unsigned long long ga = 0ull, ua = 0ull;
#pragma unroll
    for (int g = 0; g < GPL; ++g) {
        ga = group_fma2(*reinterpret_cast<const uint16_t *>(gb + 2 + 2 * (g0 + g)), &xp[4 * g], tabc, ga);
        ua = group_fma2(*reinterpret_cast<const uint16_t *>(ub + 2 + 2 * (g0 + g)), &xp[4 * g], tabc, ua);
    }
    gv = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(gb)) * hsum2(ga);
    uv = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(ub)) * hsum2(ua);
}

// h = silu(g) * u from the per-half partial sums of one row pair ([half][gate, up])
template <int SPLIT>
__device__ __forceinline__ float swiglu_part(const float *p) {
    float gv = p[0], uv = p[1];
    if (SPLIT == 2) { gv += p[2]; uv += p[3]; }
    return silu(gv) * uv;
}

// One row of a down tile (rows of I values stored back to back from a block boundary), LPR
// lanes per row, GPL groups per lane; hp = the lane's 8*GPL values of h as packed f32 pairs.
// Every lane of the LPR-group returns the full dot product.
template <int GPL, int LPR>
__device__ __forceinline__ float down_row(const uint8_t *tile, int rr, int I, int sl, const unsigned long long *hp,
                                          const uint4 *tabc) {
    const int gtile = rr * (I / 8) + sl * GPL;  // group index inside the tile
    const uint8_t *blk = tile + (gtile >> 5) * kBlockBytes;
    const int g0 = gtile & 31;
    unsigned long long acc = 0ull;
#pragma unroll
    for (int g = 0; g < GPL; ++g)
        acc = group_fma2(*reinterpret_cast<const uint16_t *>(blk + 2 + 2 * (g0 + g)), &hp[4 * g], tabc, acc);
    const float d = fp16_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
    return group_sum<LPR>(d * hsum2(acc));
}

// sum_k w_k * o_k in selection order (o_k at o[k * stride])
__device__ __forceinline__ float ordered_combine(const float *w, const float *o, int stride, int K) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (k < K) acc = fmaf(w[k], o[k * stride], acc);
    return acc;
}

}  // namespace rl
