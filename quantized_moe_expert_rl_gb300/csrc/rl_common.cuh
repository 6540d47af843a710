// rl_common.cuh - shared device helpers and host-side argument checks of librlmoe.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rl_moe.h"

namespace rl {

constexpr int kBlockValues = 256;
constexpr int kBlockBytes = 66;
constexpr int kGridBytes = 256 * 8;
constexpr unsigned kFull = 0xffffffffu;
// largest top_k * inter of a supported shape (check_shape refuses more)
constexpr int kMaxKxI = 16384;
// Bounded on-chip waits: try_wait suspends for a hardware-defined slice, so this cap is
// far beyond any legitimate wait (seconds) yet finite.
constexpr uint32_t kWaitCap = 1u << 24;

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
rl_status fail(rl_status st, const char *fmt, ...);
rl_status check_launch(const char *what);
rl_status check_shape(const rl_moe_shape *shp);
__host__ __device__ inline size_t matrix_bytes(int rows, int cols) { return (size_t)rows * cols / kBlockValues * kBlockBytes; }
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }
// cuTensorMapEncodeTiled, from the driver through the runtime (no link to the driver library);
// NULL when the driver does not provide it
inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}
// opt a kernel into more than 48 KB of dynamic shared memory (idempotent)
rl_status allow_smem(const void *kernel, size_t bytes);
// streaming multiprocessors of the current device (cached)
int sm_count();

// Launch as a programmatic dependent of the previous kernel in the stream: the kernel may
// start while its predecessor runs and must call griddepcontrol.wait before touching
// anything the predecessor writes.
template <typename Kern, typename... Args>
rl_status launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const char *what,
                     Args... args) {
    rl_status st = allow_smem((const void *)kernel, smem);
    if (st != RL_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) return fail(RL_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return RL_OK;
}

// ------------------------------------------------------------------------------------------
// device side
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int ld_ctrl(const int32_t *p) {
    return *reinterpret_cast<const volatile int32_t *>(p);
}
__device__ __forceinline__ void dev_error(int32_t *ctrl, int bits) { atomicOr(ctrl + 1, bits); }

// CTA barrier that also rejoins every warp.  A warp whose lanes took different paths (one lane
// waiting on a flag, a lane-dependent branch) can stay split long after the branch, across
// __syncthreads and across shuffles, and then each of its shuffles and votes is about thirty
// times slower (measured on GB300: ~220 cycles instead of ~7).  Only __syncwarp joins its lanes
// again, so the hot loops end every lane-dependent branch with one.  Every thread of the CTA
// must take part (no lane may have exited).
__device__ __forceinline__ void cta_sync() {
    __syncthreads();
    __syncwarp();
}
__device__ __forceinline__ int cta_sync_or(int pred) {
    const int r = __syncthreads_or(pred);
    __syncwarp();
    return r;
}

// 64-bit integer <-> f32 conversions built from 32-bit ones: the native 64-bit conversions
// run on a slow pipe here (about 100 cycles per warp instruction, measured).
// f32 of a 64-bit integer: exact up to 2^24 in magnitude, within 2^-23 relative beyond
// (deterministic, not always the correctly rounded value).
__device__ __forceinline__ float ll_to_float(long long v) {
    const unsigned long long a = v < 0 ? 0ull - (unsigned long long)v : (unsigned long long)v;
    const float m = fmaf(__uint2float_rn((uint32_t)(a >> 32)), 4294967296.0f, __uint2float_rn((uint32_t)a));
    return v < 0 ? -m : m;
}
// The integer nearest f (ties to even), for |f| < 2^55: the same value as __float2ll_rn.  Beyond
// 2^31 an f32 is an integer, so its upper and lower parts convert exactly.
__device__ __forceinline__ long long float_to_ll(float f) {
    if (fabsf(f) < 2147483648.0f) return (long long)__float2int_rn(f);
    const int hi = __float2int_rz(f * 5.9604644775390625e-8f);  // f / 2^24, toward zero
    const int lo = __float2int_rn(fmaf(-(float)hi, 16777216.0f, f));
    return (long long)hi * 16777216ll + lo;
}

// dst[j] = src[j] for j < n (16-byte items) by the whole block, four loads in flight per
// thread before their stores: a source across the host link takes microseconds per load, so
// one load at a time per thread leaves the link mostly idle.
__device__ __forceinline__ void copy16_batched(uint4 *__restrict__ dst, const uint4 *__restrict__ src, uint32_t n) {
    for (uint32_t j = threadIdx.x; j < n; j += 4 * blockDim.x) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t jj = j + u * blockDim.x;
            if (jj < n) v[u] = src[jj];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t jj = j + u * blockDim.x;
            if (jj < n) dst[jj] = v[u];
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
// sum over aligned groups of `width` lanes (width a power of two <= 32)
template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)bits));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// explicit shared-memory loads at a shared-window address (never resolved as generic loads)
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// ---- mbarrier + bulk async copy (global -> this CTA's shared memory) ----------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for phase `parity` of an mbarrier; false when the cap ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t cap = kWaitCap) {
    for (uint32_t i = 0; i < cap; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Non-blocking probe of phase `parity` (mbarrier.test_wait never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kSpinPolls = 1u << 26;  // test_wait polls (tens of cycles each): about a second
// Bounded spin on test_wait by lane 0 of the warp (the other lanes park in __syncwarp): for
// the hand-offs of a pipeline, where the wake-up delay of a suspended try_wait is too long.
// Call with the whole warp; the result is warp-uniform.
__device__ __forceinline__ bool mbar_spin_warp(uint64_t *bar, uint32_t parity, uint32_t cap = kSpinPolls) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) {
        for (uint32_t i = 0; i < cap; ++i)
            if (mbar_test_wait(bar, parity)) {
                ok = 1;
                break;
            }
    }
    __syncwarp();  // rejoin the warp (see cta_sync)
    return __shfl_sync(kFull, ok, 0) != 0;
}
// The same wait made by lane 0 of the warp alone while the other lanes park in __syncwarp, so
// that a waiting warp does not keep the shared-memory pipe busy with polls (which slows the
// warps that compute).  Call with the whole warp; the result is warp-uniform.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint32_t cap = kWaitCap) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, cap) ? 1 : 0;
    __syncwarp();  // rejoin the warp (see cta_sync)
    return __shfl_sync(kFull, ok, 0) != 0;
}
// Contiguous copy of `bytes` (multiple of 16, both addresses 16-byte aligned) into shared
// memory; completion is signalled as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// 2-D tensor copy of one box of `map` at element coordinates (x, y) into shared memory;
// completion is signalled as transaction bytes on `bar`.  x times the element size must be a
// multiple of 16 bytes; rows and columns outside the tensor read as zeros.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_l2_bulk(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// ---- the quantized block format -----------------------------------------------------------
// Dot product of `ngroups` consecutive 8-value groups of one block with 8*ngroups values of
// v (registers), without the block scale d:  sum_g sum_j grid[idx_g][j] * (+-1) * v[8g+j].
// `blk` points at the block (bytes 0-1 = d), `g0` is the first group index in the block.
template <int NG>
__device__ __forceinline__ float groups_dot(const uint8_t *blk, int g0, const float *v, const int8_t *grid_s) {
    float acc = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const uint32_t w = *reinterpret_cast<const uint16_t *>(blk + 2 + 2 * (g0 + g));
        const uint32_t idx = w & 0xffu, sg = w >> 8;
        const uint2 q = *reinterpret_cast<const uint2 *>(grid_s + 8 * idx);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t word = j < 4 ? q.x : q.y;
            float m = (float)(int8_t)((word >> (8 * (j & 3))) & 0xffu);
            m = ((sg >> j) & 1u) ? -m : m;
            acc = fmaf(m, v[8 * g + j], acc);
        }
    }
    return acc;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace rl
