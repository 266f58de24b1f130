// kda_device.cuh -- device helpers shared by the KDA kernels (sm_103a): bf16 conversion, mbarrier and
// bulk-copy (TMA) wrappers written as inline PTX, bounded waits, deterministic warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Give up on an asynchronous copy after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }
// Fast-division variant for the output gate, which only scales a bf16 output.
__device__ __forceinline__ float sigmoid_gate(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive once and announce `bytes` of transactions for the current phase (0 completes a bare arrive).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.  16-byte aligned addresses,
// size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy shared -> global (TMA engine), tracked as a bulk async-group of the issuing thread.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the sources of this thread's committed bulk groups have been read (smem reusable).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until this thread's committed bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase of `bar` with the given parity; gives up after limit_ns and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Deterministic sum of x[0..n) by one full warp (lane-strided partials, then a fixed xor tree).
__device__ __forceinline__ float warp_sum_array(const float *x, int n) {
    const int lane = threadIdx.x & 31;
    float s = 0.f;
    for (int i = lane; i < n; i += 32) s += x[i];
    return warp_sum(s);
}

__device__ __forceinline__ float warp_dot_array(const float *x, const float *y, int n) {
    const int lane = threadIdx.x & 31;
    float s = 0.f;
    for (int i = lane; i < n; i += 32) s = fmaf(x[i], y[i], s);
    return warp_sum(s);
}

// Pool state element access for an fp32 or a bf16 pool (bf16: round to nearest even on store).
__device__ __forceinline__ float load_state(const void *S, bool bf, size_t idx) {
    return bf ? bf2f(reinterpret_cast<const uint16_t *>(S)[idx]) : reinterpret_cast<const float *>(S)[idx];
}
__device__ __forceinline__ void store_state(void *S, bool bf, size_t idx, float v) {
    if (bf)
        reinterpret_cast<uint16_t *>(S)[idx] = f2bf(v);
    else
        reinterpret_cast<float *>(S)[idx] = v;
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

}  // namespace kda
