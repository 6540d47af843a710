// fill.cu - the fill of a layer's absent selected experts done by the GPU itself.
//
// Red Lite dev23 - per-layer early-out, "What changed" item 1: when a layer selects experts
// that are not resident, their records are loaded and the layer runs with the experts the
// router picked.  Done from the host, that costs a round trip per layer (read the flag and the
// selections, copy, re-resolve, resume).  Here the device finds the missing experts in the
// selection, copies their records from a source it can read (a pinned host backing store, read
// over the host link) into their HBM slots, marks them resident, re-resolves the layer's slots
// and clears the layer's early-out flag, so the next kernels of the stream run the layer with
// no host involvement.  The per-layer miss counts written by rl_route are left as they are.
//
//   mark:     every selection (t, k) of the layer whose slot is 0 claims its expert once
//             (need[e]) and appends it to a list of the experts to copy
//   copy:     a fixed grid walks (listed expert, 16 KB chunk) pairs and copies the records
//   finalize: residency[layer][e] = dst for each listed expert, *filled += count; then the
//             layer is recorded in *first_early_out, ctrl[0] cleared, the list emptied
//   resolve:  slots[t][k] = residency[layer][ids[t][k]]
#include <algorithm>

#include "rl_common.cuh"

namespace rl {

constexpr int kFillChunk = 16384;  // bytes per (expert, chunk) work item

struct FillWs {  // [count (256 B) | need u32[E] | list i32[E]]
    size_t need, list, total;
    explicit FillWs(int E) {
        need = 256;
        list = need + align_up((size_t)E * sizeof(uint32_t), 256);
        total = list + align_up((size_t)E * sizeof(int32_t), 256);
    }
};

__global__ void __launch_bounds__(256) fill_mark_kernel(const int32_t *__restrict__ ids,
                                                        const uint64_t *__restrict__ slots, uint32_t *count,
                                                        uint32_t *need, int32_t *list, int n, int E) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int e = ids[i];
        if (slots[i] == 0 && e >= 0 && e < E && atomicExch(need + e, 1u) == 0u) list[atomicAdd(count, 1u)] = e;
    }
}

__global__ void __launch_bounds__(256) fill_copy_kernel(const uint32_t *__restrict__ count,
                                                        const int32_t *__restrict__ list,
                                                        const uint64_t *__restrict__ src,
                                                        const uint64_t *__restrict__ dst, int chunks,
                                                        uint32_t rec_bytes) {
    const int items = (int)*count * chunks;
    for (int w = blockIdx.x; w < items; w += gridDim.x) {
        const int e = list[w / chunks], c = w % chunks;
        const uint64_t s = src[e], d = dst[e];
        if (s == 0 || d == 0 || ((s | d) & 15)) continue;  // finalize reports it
        const uint32_t lo = (uint32_t)c * kFillChunk, hi = min(rec_bytes, lo + (uint32_t)kFillChunk);
        copy16_batched(reinterpret_cast<uint4 *>(d + lo), reinterpret_cast<const uint4 *>(s + lo), (hi - lo) / 16);
    }
}

__global__ void __launch_bounds__(512) fill_finalize_kernel(uint32_t *count, uint32_t *need, const int32_t *list,
                                                            const uint64_t *__restrict__ src,
                                                            const uint64_t *__restrict__ dst, uint64_t *table_row,
                                                            uint32_t *filled, int32_t *first_early_out, int32_t *ctrl,
                                                            int layer) {
    const int n = (int)*count;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int e = list[i];
        need[e] = 0u;
        const uint64_t s = src[e], d = dst[e];
        if (s == 0 || d == 0) {
            dev_error(ctrl, RL_DEVERR_MISSING);
        } else if ((s | d) & 15) {
            dev_error(ctrl, RL_DEVERR_SLOT_ALIGN);
        } else {
            table_row[e] = d;
            atomicAdd(filled, 1u);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && n > 0) {
        atomicMin(first_early_out, layer);
        if (ctrl[0] == layer) ctrl[0] = RL_NO_EARLY_OUT;
        *count = 0u;
    }
}

__global__ void fill_resolve_kernel(const int32_t *__restrict__ ids, const uint64_t *__restrict__ table_row,
                                    uint64_t *slots, int n, int E) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int e = ids[i];
        slots[i] = (e >= 0 && e < E) ? table_row[e] : 0;
    }
}

}  // namespace rl

using namespace rl;

extern "C" size_t rl_fill_workspace_bytes(const rl_moe_shape *shp) {
    if (!shp || shp->n_experts <= 0) return 0;
    return FillWs(shp->n_experts).total;
}

extern "C" rl_status rl_host_device_pointer(const void *host, uint64_t *device) {
    if (!host || !device) return fail(RL_ERR_INVALID, "rl_host_device_pointer: NULL argument");
    void *d = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void *>(host), 0);
    if (e != cudaSuccess || !d) {
        (void)cudaGetLastError();
        return fail(RL_ERR_INVALID, "rl_host_device_pointer: %p is not page-locked host memory the device can read (%s)",
                    host, cudaGetErrorString(e));
    }
    *device = reinterpret_cast<uint64_t>(d);
    return RL_OK;
}

extern "C" rl_status rl_fill_missing(const rl_moe_shape *shp, int32_t layer, int32_t T, const int32_t *ids,
                                     uint64_t *slots, uint64_t *residency, const uint64_t *src, const uint64_t *dst,
                                     uint32_t *filled, int32_t *first_early_out, int32_t *ctrl, void *ws,
                                     size_t ws_bytes, void *stream) {
    rl_status st = check_shape(shp);
    if (st != RL_OK) return st;
    if (layer < 0 || layer >= shp->n_layers)
        return fail(RL_ERR_INVALID, "rl_fill_missing: layer %d outside [0,%d)", layer, shp->n_layers);
    if (T < 0 || !ids || !slots || !residency || !src || !dst || !filled || !first_early_out || !ctrl)
        return fail(RL_ERR_INVALID, "rl_fill_missing: bad arguments");
    const int E = shp->n_experts;
    const FillWs W(E);
    if (!ws || ws_bytes < W.total)
        return fail(RL_ERR_INVALID, "rl_fill_missing: workspace of %zu B needed, %zu given", W.total, ws_bytes);
    if (reinterpret_cast<uintptr_t>(ws) & 15) return fail(RL_ERR_INVALID, "rl_fill_missing: ws must be 16-byte aligned");
    const size_t rb = 3 * matrix_bytes(shp->inter, shp->hidden);
    if (rb % 16 != 0 || rb > 0xffffffffull)
        return fail(RL_ERR_UNSUPPORTED, "rl_fill_missing: record of %zu B is not a 16-byte multiple", rb);
    if ((long long)T * shp->top_k > (1ll << 30)) return fail(RL_ERR_UNSUPPORTED, "rl_fill_missing: too many selections");
    const int n = T * shp->top_k;
    if (n == 0) return RL_OK;
    cudaStream_t s = as_stream(stream);
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint32_t *count = reinterpret_cast<uint32_t *>(w8);
    uint32_t *need = reinterpret_cast<uint32_t *>(w8 + W.need);
    int32_t *list = reinterpret_cast<int32_t *>(w8 + W.list);
    const size_t off = (size_t)layer * E;
    const int chunks = (int)((rb + kFillChunk - 1) / kFillChunk);
    const int grid = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
    fill_mark_kernel<<<grid, 256, 0, s>>>(ids, slots, count, need, list, n, E);
    fill_copy_kernel<<<2 * sm_count(), 256, 0, s>>>(count, list, src + off, dst + off, chunks, (uint32_t)rb);
    fill_finalize_kernel<<<1, 512, 0, s>>>(count, need, list, src + off, dst + off, residency + off, filled,
                                           first_early_out, ctrl, layer);
    fill_resolve_kernel<<<grid, 256, 0, s>>>(ids, residency + off, slots, n, E);
    return check_launch("rl_fill_missing");
}
