// prefill_common.cuh - argument checks, workspace layout and the ordered combine shared by
// the two grouped prefill paths (tensor-core f16 and CUDA-core f32).
#pragma once
#include "rl_common.cuh"

namespace rl {

struct PrefillArgs {
    int layer, T, H, E, K, I, P, accumulate;
    const float *xn;
    const uint32_t *offs, *pair_tok;
    const uint8_t *pair_k;
    const uint64_t *slots;
    const float *weights;
    const int8_t *codebook;
    float *y;
    int32_t *ctrl;
    // workspace carve-up
    float *hbuf;              // [P][I]   f32 SwiGLU activations, pair order (f32 path)
    float *outbuf;            // [T*K][H] f32 expert outputs, indexed by (token, k)
    uint16_t *xb16;           // [P'][H]  f16 copy of xn gathered in pair order (tensor-core path)
    uint16_t *hb16;           // [P'][I]  f16 SwiGLU activations, pair order (tensor-core path)
    void *units;              // tensor-core work-unit lists
};

// P' = max(P, 16): the tensor-core path reads its 16-bit operands in boxes of 16 pair rows
struct PrefillWs {
    size_t h, out, xb, hb, units, total;
    PrefillWs(int T, int H, int K, int I, int E) {
        const size_t P = (size_t)T * K, P16 = P > 16 ? P : 16;
        h = align_up(P * I * sizeof(float), 256);
        out = align_up(P * H * sizeof(float), 256);
        xb = align_up(P16 * H * 2, 256);
        hb = align_up(P16 * I * 2, 256);
        // unit lists: at most (P / 128 + E) token blocks x (I / 64 gate/up + H / 128 down) row tiles
        units = align_up(256 + 4 * (P / 128 + (size_t)E) * ((size_t)I / 64 + (size_t)H / 128), 256);
        total = h + out + xb + hb + units;
    }
};

rl_status prefill_check(const rl_moe_shape *shp, int32_t layer, int32_t T, const float *xn, const uint32_t *offs,
                        const uint32_t *pair_tok, const uint8_t *pair_k, const uint64_t *slots,
                        const float *weights, const int8_t *codebook, float *y, int32_t accumulate,
                        int32_t *ctrl, void *ws, size_t ws_bytes, const char *who, PrefillArgs *a);
rl_status launch_ordered_sum(const PrefillArgs &a, cudaStream_t s);

}  // namespace rl
