// abi.cu - host-side status reporting, shape checks and small ABI queries of librlmoe.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <map>
#include <utility>

#include "rl_common.cuh"

namespace rl {

static thread_local char g_last_error[512] = "";

rl_status fail(rl_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

rl_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return RL_OK;
}

rl_status check_shape(const rl_moe_shape *shp) {
    if (!shp) return fail(RL_ERR_INVALID, "shape pointer is NULL");
    const int H = shp->hidden, E = shp->n_experts, K = shp->top_k, I = shp->inter, L = shp->n_layers;
    if (H <= 0 || E <= 0 || K <= 0 || I <= 0 || L <= 0)
        return fail(RL_ERR_INVALID, "shape fields must be positive (H=%d E=%d K=%d I=%d L=%d)", H, E, K, I, L);
    if (!(H == 256 || H == 512 || H == 1024 || H == 2048))
        return fail(RL_ERR_UNSUPPORTED, "hidden=%d: supported 256, 512, 1024, 2048", H);
    if (!(I == 128 || I == 256 || I == 512 || I == 1024 || I == 2048))
        return fail(RL_ERR_UNSUPPORTED, "inter=%d: supported 128, 256, 512, 1024, 2048", I);
    if (K > 16) return fail(RL_ERR_UNSUPPORTED, "top_k=%d > 16", K);
    if (E > 512) return fail(RL_ERR_UNSUPPORTED, "n_experts=%d > 512", E);
    if (K > E) return fail(RL_ERR_INVALID, "top_k=%d > n_experts=%d", K, E);
    if ((size_t)K * I > (size_t)kMaxKxI) return fail(RL_ERR_UNSUPPORTED, "top_k*inter=%d > %d", K * I, kMaxKxI);
    return RL_OK;
}

// The attribute belongs to the kernel on the current device, so the cache is per device: a
// process that drives several GPUs sets it once on each.
rl_status allow_smem(const void *kernel, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(dev, kernel);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return RL_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "cudaFuncSetAttribute(%zu B smem): %s", bytes, cudaGetErrorString(e));
    done[key] = bytes;
    return RL_OK;
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace rl

extern "C" int32_t rl_abi_version(void) { return RL_ABI_VERSION; }

extern "C" const char *rl_last_error(void) { return rl::g_last_error; }

extern "C" size_t rl_record_bytes(const rl_moe_shape *shp) {
    if (!shp || shp->hidden <= 0 || shp->inter <= 0 || ((size_t)shp->hidden * shp->inter) % 256 != 0) return 0;
    return 3 * rl::matrix_bytes(shp->inter, shp->hidden);
}
