// prefill_tc.cu - grouped expert GEMMs of a prefill chunk on the tcgen05 tensor cores.
#include "prefill_common.cuh"

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
    (void)stream;
    return fail(RL_ERR_UNSUPPORTED, "moe_prefill_chunk: tensor-core path not built yet");
}
